// Backward preparation: transpose, sort, run-length encoding (kimbodo
// "Kimbodo Engineering Perspective" names these three steps; kimbodo "What
// Happened": updates are grouped by (table, row)).
//
//  1. bag_marks_kernel + keys_kernel: one (table,row) key per lookup, key =
//     rowbase_t + idx (or the sentinel sum-of-rows for an index out of
//     range), and its sort value: with per-lookup scales (weights or mean
//     pooling) the position, and the bag and scale s_i by position; without,
//     the flat bag itself (the apply then needs nothing else).  Also the
//     first radix pass's digit counts.
//     Positions are tiled evenly (the first bag of each tile is marked by a
//     pass over the bags), so bag lengths do not unbalance the work.
//  2. a stable LSD radix sort of (key, value), 8- or 9-bit digits,
//     reduce-then-scan per pass: per-tile digit counts and the pass's digit
//     histogram (the keys kernel gives the first pass's, the upsweep the
//     others), a scan per digit over the tiles, and a scatter that
//     ranks each tile's keys by digit (warp match of equal digits + per-warp
//     counters, in input order) and writes each digit's run contiguously.
//  3. run-length encoding, reduce-then-scan: runs per tile
//     (rle_count_kernel), a scan over the tiles, then rle_kernel writes the
//     distinct keys with their first sorted slot (runstart[U] = N) and the
//     first distinct key of each table.
//  4. chunk_count/chunk_write: number the chunks (256 to 1024 lookups, by
//     batch size) of every run of at least kLongRun lookups in key order (a
//     scan over the distinct keys), so each table's chunks form one
//     consecutive range for the apply step.
#include "tbe_internal.cuh"

namespace tbe {

// ---------------------------------------------------------------- block scan

// Exclusive scan of one value per thread over a 256-thread block; returns the
// exclusive prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan_256(uint32_t v, uint32_t* s_warp,
                                                             uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < 8 ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < 8) s_warp[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t warp_excl = warp == 0 ? 0u : s_warp[warp - 1];
    const uint32_t tot = s_warp[7];
    __syncthreads();  // s_warp may be reused by the caller
    *total = tot;
    return warp_excl + x - v;
}

// Exclusive scan of n counts in place by one block of THREADS threads, each
// thread taking a contiguous chunk (one block-wide scan in all), plus
// `start`; returns the total on every thread.
template <int THREADS>
__device__ __forceinline__ uint32_t block_scan_row(uint32_t* __restrict__ row, uint32_t n, uint32_t start,
                                                   uint32_t* s_warp) {
    constexpr int WARPS = THREADS / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t chunk = (n + THREADS - 1) / THREADS;
    const uint32_t i0 = tid * chunk, i1 = tmin<uint32_t>(i0 + chunk, n);
    uint32_t sum = 0;
    for (uint32_t i = i0; i < i1; ++i) sum += row[i];
    uint32_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        const uint32_t c = s_warp[w];
        if (w < warp) before += c;
        total += c;
    }
    uint32_t run = start + before + x - sum;
    for (uint32_t i = i0; i < i1; ++i) {
        const uint32_t c = row[i];
        row[i] = run;
        run += c;
    }
    return start + total;
}

__device__ __forceinline__ uint32_t block_scan_row_1024(uint32_t* __restrict__ row, uint32_t n, uint32_t start,
                                                        uint32_t* s_warp) {
    return block_scan_row<1024>(row, n, start, s_warp);
}

// ------------------------------------------------------------------ keys

constexpr int kKeysWindow = kSortTile + 1;  // offsets staged per tile

// Largest k in [0, nbags] with off[k] <= p, found by the whole block: each
// round the threads test evenly spaced candidates of the remaining interval
// and a block-wide count of "off[k] <= p" narrows it 256-fold, so two million
// bags take three rounds of one load each.  Malformed (non-monotone) offsets
// give some in-range answer.
template <typename IDX>
__device__ __forceinline__ int64_t block_find_bag(const IDX* off, int64_t nbags, int64_t p) {
    int64_t lo = 0, hi = nbags + 1;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const int64_t step = (hi - lo + blockDim.x - 1) / blockDim.x;
        const int64_t k = lo + (int64_t)threadIdx.x * step;
        const bool pred = k < hi && ld_index(off, k) <= p;
        const int c = __syncthreads_count(pred);
        const int64_t nlo = lo + (int64_t)(c > 0 ? c - 1 : 0) * step;
        const int64_t nhi = tmin<int64_t>(hi, lo + (int64_t)(c > 0 ? c : 1) * step);
        lo = nlo;
        hi = tmax<int64_t>(nhi, nlo + 1);
    }
    return lo;
}

template <typename IDX>
__device__ __forceinline__ int64_t upper_bound_global(const IDX* off, int64_t lo, int64_t hi, int64_t p) {
    // first k in [lo, hi) with off[k] > p (hi if none)
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (ld_index(off, mid) > p)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// Offsets check, the first position of every table (tpos) and the first bag
// of every key tile: a grid-stride pass over the bags; a bag [o, o1) marks
// every tile whose first position it holds, so with valid offsets each tile
// start is marked exactly once (by the bag that contains it).  Malformed offsets leave some marks stale or zero; the keys
// kernel only uses marks to narrow its search and stays in range regardless.
template <typename IDX>
__global__ void __launch_bounds__(256) bag_marks_kernel(PrepArgs a, Workspace ws) {
    chain_wait();

    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const int64_t nbags = (int64_t)a.T * a.B;
    uint32_t err = 0;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g <= nbags;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = ld_index(off, g);
        if (o < 0 || o > a.N) err |= ERR_OFFSETS;
        if (g == 0 && o != 0) err |= ERR_OFFSETS;
        if (g == nbags && o != a.N) err |= ERR_OFFSETS;
        const uint32_t oc = (uint32_t)tmin<int64_t>(tmax<int64_t>(o, 0), a.N);
        const int tg = (int)(g / a.B), bl = (int)(g % a.B);
        if (bl == 0) ws.tpos[tg] = oc;  // table starts
        if (a.compact) {                // bag offsets of the dense tables
            if (tg < a.T && a.tabs[tg].dslot >= 0) ws.dboff[(int64_t)a.tabs[tg].dslot * (a.B + 1) + bl] = oc;
            if (bl == 0 && tg > 0 && a.tabs[tg - 1].dslot >= 0)
                ws.dboff[(int64_t)a.tabs[tg - 1].dslot * (a.B + 1) + a.B] = oc;
        }
        if (g < nbags) {
            const int64_t o1 = ld_index(off, g + 1);
            if (o1 < o) err |= ERR_OFFSETS;
            if (o >= 0 && o < o1 && o1 <= a.N)
                for (int64_t q = (o + kSortTile - 1) / kSortTile; q * kSortTile < o1; ++q)
                    ws.tile_bag[q] = (uint32_t)g;
        }
    }
    if (err) atomicOr(&a.blk->error, err);
}

// Where each sorted-path table's keys go when dense tables are present (their
// lookups are not sorted): cbase[t] = the lookups of the sorted-path tables
// before t, cbase[T] and counters[CTR_NS] = all of them (one CTA).
__global__ void __launch_bounds__(1024) compact_kernel(PrepArgs a, Workspace ws) {
    chain_wait();

    __shared__ uint32_t s_warp[32];
    for (int t = threadIdx.x; t < a.T; t += blockDim.x) {
        uint32_t c = 0;
        if (a.tabs[t].dslot < 0) {
            const uint32_t lo = ws.tpos[t];
            c = tmax<uint32_t>(ws.tpos[t + 1], lo) - lo;
        }
        ws.cbase[t] = c;
    }
    __syncthreads();
    const uint32_t total = tmin<uint32_t>(block_scan_row_1024(ws.cbase, (uint32_t)a.T, 0u, s_warp), (uint32_t)a.N);
    if (threadIdx.x == 0) {
        ws.cbase[a.T] = total;
        ws.counters[CTR_NS] = total;
    }
}

// Keys to sort: all lookups, or those of the sorted-path tables when dense
// tables are present.
__device__ __forceinline__ uint32_t sorted_count(const PrepArgs& a, const Workspace& ws) {
    return ws.compact ? tmin<uint32_t>(ws.counters[CTR_NS], (uint32_t)a.N) : (uint32_t)a.N;
}

// One key per position, tile by tile.  The tile's bags [bf, bl] come from
// the marks (the last tile finds its last bag with a block-wide search);
// their offsets are staged in shared memory and every position learns its bag
// from the bag starts: each non-empty bag marks its first position in the
// tile, and a position's bag is the last mark at or before it (per 32
// positions a ballot of the marks, the highest marked lane at or below each
// lane, and a carry from the previous 32).  Warp w takes positions
// w*512 + k*32 + lane (k < 16), so loads and stores are coalesced.  The first
// radix pass's digit counts are kept per tile (for the sort's scan) and per
// block (added to the first pass's global histogram at the end); the later
// passes count their digits in the upsweep.
template <typename IDX>
__global__ void __launch_bounds__(256, 3) keys_kernel(PrepArgs a, Workspace ws) {
    chain_wait();

    __shared__ int32_t s_off[kKeysWindow + 3];  // offsets bf .. bl+1 (N < 2^30)
    __shared__ int16_t s_mark[kSortTile];       // window index of the bag starting at each position
    __shared__ float s_w[kSortTile];            // the tile's per-sample weights
    __shared__ uint32_t s_hist0[kMaxRadix];  // first-pass digit histogram of the block
    __shared__ uint32_t s_tc[kMaxRadix];  // first-pass digit counts of the current tile
    __shared__ int32_t s_wlast[kSortThreads / 32];
    __shared__ int64_t s_last;
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const int64_t nbags = (int64_t)a.T * a.B;
    const int dbits = a.digit_bits;
    const uint32_t dmask = (1u << dbits) - 1u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t Nc = a.N;  // offsets are clamped to [0, N] when staged
    const uint32_t ns = tmax<uint32_t>(sorted_count(a, ws), 1u);
    uint32_t err = 0;

    for (int i = threadIdx.x; i < kMaxRadix; i += blockDim.x) s_hist0[i] = 0;
    for (int i = threadIdx.x; i < kMaxRadix; i += blockDim.x) s_tc[i] = 0;

    const int64_t tiles = (a.N + kSortTile - 1) / kSortTile;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t p0 = tile * kSortTile;
        const int64_t p1 = min(p0 + (int64_t)kSortTile, a.N);
        const int n = (int)(p1 - p0);
        __syncthreads();  // the previous tile is done with the shared arrays
        const int64_t bf = tmin<int64_t>((int64_t)__ldg(ws.tile_bag + tile), nbags - 1);
        int64_t bl;
        if (tile + 1 < tiles) {
            bl = tmin<int64_t>(tmax<int64_t>((int64_t)__ldg(ws.tile_bag + tile + 1), bf), nbags - 1);
        } else {
            const int64_t l = block_find_bag(off, nbags, p1 - 1);
            if (threadIdx.x == 0) s_last = l;
            __syncthreads();
            bl = tmin<int64_t>(tmax<int64_t>(s_last, bf), nbags - 1);
        }
        const int64_t nwin = bl - bf + 2;  // offsets bf .. bl+1
        const bool staged = nwin <= kKeysWindow;
        // the tile's indices and weights, loaded before the bag map is built
        // (the weights into shared memory, read after the next sync)
        IDX xv[kSortItems];
#pragma unroll
        for (int k = 0; k < kSortItems; ++k) {
            const int li = warp * (32 * kSortItems) + k * 32 + lane;
            xv[k] = li < n ? ind[p0 + li] : (IDX)0;
        }
        if (ws.scale && a.weights) {
#pragma unroll 4
            for (int i = threadIdx.x; i < n; i += kSortThreads) s_w[i] = __ldg(a.weights + p0 + i);
            __syncthreads();
        }
        // window index of each item's bag (staged tiles), two per register
        uint32_t bj2[kSortItems / 2] = {};
        auto bj_get = [&](int q) -> int { return (int)((bj2[q >> 1] >> (16 * (q & 1))) & 0xffffu); };
        auto bj_set = [&](int q, int v) {
            const uint32_t h = (uint32_t)v & 0xffffu;
            bj2[q >> 1] = (q & 1) ? ((bj2[q >> 1] & 0x0000ffffu) | (h << 16)) : ((bj2[q >> 1] & 0xffff0000u) | h);
        };
        if (staged) {
            for (int64_t k = threadIdx.x; k < nwin; k += blockDim.x)
                s_off[k] = (int32_t)tmin<int64_t>(tmax<int64_t>(ld_index(off, bf + k), 0), Nc);
#pragma unroll
            for (int k = 0; k < kSortItems; ++k) s_mark[k * kSortThreads + threadIdx.x] = -1;
            __syncthreads();
            // each non-empty bag marks its first position inside the tile
            // (with valid offsets no two bags mark the same position)
            for (int j = threadIdx.x; j < (int)nwin - 1; j += blockDim.x) {
                const int64_t st = s_off[j];
                if (st < s_off[j + 1] && st >= p0 && st < p1) s_mark[st - p0] = (int16_t)j;
            }
            __syncthreads();
            // last mark at or before each position, per warp over its 512
            int carry = -1;
#pragma unroll
            for (int k = 0; k < kSortItems; ++k) {
                const int m = s_mark[warp * (32 * kSortItems) + k * 32 + lane];
                const uint32_t marked = __ballot_sync(0xffffffffu, m >= 0);
                const uint32_t upto = marked & (0xffffffffu >> (31 - lane));
                const int v = __shfl_sync(0xffffffffu, m, upto ? 31 - __clz(upto) : 0);
                bj_set(k, upto ? v : carry);  // -1 (no mark yet) is kept as 0xffff
                const int top = __shfl_sync(0xffffffffu, m, marked ? 31 - __clz(marked) : 0);
                carry = marked ? top : carry;
            }
            if (lane == 0) s_wlast[warp] = carry;
            __syncthreads();
            int pre = 0;  // positions before the first mark belong to bag bf (index 0)
            for (int w = warp - 1; w >= 0; --w)
                if (s_wlast[w] >= 0) {
                    pre = s_wlast[w];
                    break;
                }
#pragma unroll
            for (int k = 0; k < kSortItems; ++k) {
                const int b = bj_get(k);
                bj_set(k, tmin<int>(b == 0xffff ? pre : b, (int)nwin - 2));
            }
        }
        // table of each bag: the window starts in table tf (whose descriptor
        // is read once per tile); a bag past it walks forward (rare).  Sizes
        // fit 32 bits: N < 2^30, T*B < 2^31, sum of rows < 2^32.
        const uint32_t B32 = (uint32_t)a.B;
        const uint32_t bf32 = (uint32_t)bf;
        const int tf = (int)(bf32 / B32);
        const uint32_t tf_end = (uint32_t)(tf + 1) * B32;  // first bag of the next table
        const uint32_t rows_f = (uint32_t)a.tabs[tf].rows;
        const uint32_t rowbase_f = (uint32_t)a.tabs[tf].rowbase;
        const bool dense_f = a.tabs[tf].dslot >= 0;
        // compacted slot of a sorted-path lookup: cbase[t] + (p - tpos[t])
        const uint32_t shift_f = ws.compact ? ws.cbase[tf] - ws.tpos[tf] : 0u;
        const uint32_t p032 = (uint32_t)p0;
#pragma unroll
        for (int k = 0; k < kSortItems; ++k) {
            const int li = warp * (32 * kSortItems) + k * 32 + lane;
            const bool valid = li < n;
            uint32_t keyk = 0xffffffffu;
            if (valid) {
                const uint32_t p = p032 + (uint32_t)li;
                uint32_t bag;
                int32_t L;
                if (staged) {
                    const int j = bj_get(k);
                    bag = bf32 + (uint32_t)j;
                    L = s_off[j + 1] - s_off[j];
                } else {
                    int64_t b = upper_bound_global(off, bf, min(bl + 2, nbags + 1), (int64_t)p) - 1;
                    b = tmax<int64_t>(tmin<int64_t>(b, nbags - 1), 0);
                    bag = (uint32_t)b;
                    L = (int32_t)(ld_index(off, b + 1) - ld_index(off, b));
                }
                uint32_t rows = rows_f, rowbase = rowbase_f, shift = shift_f;
                bool dense = dense_f;
                if (bag >= tf_end) {
                    int t = tf + 1;
                    for (uint32_t tb = tf_end + B32; bag >= tb && t < a.T - 1; tb += B32) ++t;
                    rows = (uint32_t)a.tabs[t].rows;
                    rowbase = (uint32_t)a.tabs[t].rowbase;
                    dense = a.tabs[t].dslot >= 0;
                    shift = ws.compact ? ws.cbase[t] - ws.tpos[t] : 0u;
                }
                // an index outside [0, rows) (negative ones included) is skipped
                const bool in_range = (uint64_t)(int64_t)xv[k] < (uint64_t)rows;
                if (!in_range) err |= ERR_OOB;
                if (dense) {
                    // dense tables: the row for the shared-memory backward, no
                    // key (and no bag: the dense backward walks bag offsets)
                    ws.hrow[p] = in_range ? (uint16_t)xv[k] : (uint16_t)0xffffu;
                } else {
                    const uint32_t key = in_range ? rowbase + (uint32_t)xv[k] : a.total_rows;
                    keyk = key;
                    // malformed offsets could send a slot out of range: clamp
                    const uint32_t c = ws.compact ? tmin<uint32_t>(p + shift, ns - 1u) : p;
                    ws.keys[0][c] = key;
                    if (!ws.scale) {
                        ws.vals[0][c] = bag;  // no scale to look up: the sort carries the bag itself
                    } else {
                        ws.bag[p] = bag;
                        if (ws.compact) ws.vals[0][c] = p;
                    }
                }
                if (ws.scale) {
                    float sc = a.weights ? s_w[li] : 1.f;
                    if (a.mean && L > 0) sc = __fdiv_rn(sc, (float)L);
                    ws.scale[p] = sc;
                }
            }
            // first-pass digit counts of this tile (the later passes' come
            // from the upsweep); compacted keys do not follow these tiles,
            // so then the sort counts every pass itself
            if (keyk != 0xffffffffu && !ws.compact) atomicAdd(&s_tc[keyk & dmask], 1u);
        }
        // the tile's first-pass digit counts: to the sort's count table and
        // the block's first-pass histogram
        if (!ws.compact) {
            __syncthreads();
            for (int d = threadIdx.x; d <= (int)dmask; d += blockDim.x) {
                const uint32_t c = s_tc[d];
                ws.tcount[(size_t)d * tiles + tile] = c;
                s_hist0[d] += c;
                s_tc[d] = 0;
            }
        }
    }
    if (!ws.compact) {
        __syncthreads();
        for (int d = threadIdx.x; d <= (int)dmask; d += blockDim.x)
            if (s_hist0[d]) atomicAdd(ws.hist + d, s_hist0[d]);
    }
    if (err) atomicOr(&a.blk->error, err);
}

// --------------------------------------------------------- one radix pass
//
// Reduce-then-scan: the digit counts of every tile (tcount[d][tile], digit
// major) come from the keys kernel for the first pass and from
// upsweep_kernel for later ones; scan_kernel turns each digit's row into the
// global start of that digit's keys from each tile; downsweep_kernel ranks
// each tile's keys by digit and scatters them.  Nothing waits on another
// tile, so the time per tile does not grow with the number of tiles in
// flight.

// Digit counts of tiles of keys (a CTA walks tiles blockIdx.x + k*gridDim.x),
// also summed per CTA and added once to the pass's global digit histogram.
// Only the tiles that hold keys are counted (with compacted keys the device
// count of sorted keys can be far below N); the scan and the scatter skip the
// rest too.
template <int RB>
__global__ void __launch_bounds__(kSortThreads) upsweep_kernel(const uint32_t* __restrict__ keys, uint32_t N,
                                                               const uint32_t* __restrict__ nsp, int shift,
                                                               uint32_t* __restrict__ tcount, uint32_t tiles,
                                                               uint32_t* __restrict__ hist) {
    chain_wait();

    constexpr int RADIX = 1 << RB;
    __shared__ uint32_t s_c[RADIX];
    __shared__ uint32_t s_g[RADIX];
    const int tid = threadIdx.x;
    if (nsp) N = tmin<uint32_t>(*nsp, N);  // sorted keys (device count)
    const uint32_t used = tmin<uint32_t>(tiles, (N + kSortTile - 1) / kSortTile);  // tiles holding keys
    for (int d = tid; d < RADIX; d += kSortThreads) s_c[d] = s_g[d] = 0;
    for (uint32_t tile = blockIdx.x; tile < used; tile += gridDim.x) {
        __syncthreads();  // counts of the previous tile read and cleared
        const uint32_t base = tile * kSortTile;
        uint32_t key[kSortItems];
#pragma unroll
        for (int k = 0; k < kSortItems; ++k) {
            const uint32_t idx = base + k * kSortThreads + tid;
            key[k] = idx < N ? __ldg(keys + idx) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kSortItems; ++k)
            if (base + k * kSortThreads + tid < N) atomicAdd(&s_c[(key[k] >> shift) & (RADIX - 1)], 1u);
        __syncthreads();
        for (int d = tid; d < RADIX; d += kSortThreads) {
            const uint32_t c = s_c[d];
            tcount[(size_t)d * tiles + tile] = c;
            s_g[d] += c;
            s_c[d] = 0;
        }
    }
    __syncthreads();
    for (int d = tid; d < RADIX; d += kSortThreads)
        if (s_g[d]) atomicAdd(hist + d, s_g[d]);  // the pass's global histogram
}

// Exclusive scan of one digit's row of tile counts (one CTA of THREADS per
// digit), offset by the number of keys with a smaller digit: the global
// start of the digit's keys from each tile, in place.
template <int RB, int THREADS>
__global__ void __launch_bounds__(THREADS) scan_kernel(uint32_t* __restrict__ tcount, const uint32_t* __restrict__ hist,
                                                       uint32_t tiles, uint32_t N, const uint32_t* __restrict__ nsp) {
    chain_wait();

    constexpr int WARPS = THREADS / 32;
    __shared__ uint32_t s_warp[WARPS];
    __shared__ uint32_t s_start;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = blockIdx.x;
    // keys with a smaller digit
    {
        uint32_t v = 0;
        for (int e = tid; e < d; e += THREADS) v += __ldg(hist + e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_warp[warp] = v;
        __syncthreads();
        if (tid == 0) {
            uint32_t t = 0;
            for (int w = 0; w < WARPS; ++w) t += s_warp[w];
            s_start = t;
        }
        __syncthreads();
    }
    const uint32_t start = s_start;
    __syncthreads();  // s_warp is reused below
    if (nsp) N = tmin<uint32_t>(*nsp, N);  // sorted keys (device count)
    const uint32_t used = tmin<uint32_t>(tiles, (N + kSortTile - 1) / kSortTile);  // tiles holding keys
    block_scan_row<THREADS>(tcount + (size_t)d * tiles, used, start, s_warp);
}

// Scan of every digit's row: 256-thread CTAs (all resident at once) while a
// thread's share of a row stays small, 1024-thread ones beyond.
template <int RB>
void launch_scan(uint32_t* tcount, const uint32_t* hist, uint32_t tiles, uint32_t N, const uint32_t* nsp,
                 cudaStream_t s) {
    if (tiles <= 256u * 16u || nsp)  // compacted keys: usually few of the tiles hold keys
        launch_chained(scan_kernel<RB, 256>, dim3(1 << RB), dim3(256), s, tcount, hist, tiles, N, nsp);
    else
        launch_chained(scan_kernel<RB, 1024>, dim3(1 << RB), dim3(1024), s, tcount, hist, tiles, N, nsp);
}

// Lanes of the warp holding the same digit d (RADIX, past the end, counts as a
// digit too).  MATCH: one match.any per key, fewer instructions but a longer
// latency; otherwise one ballot per bit of the (RB+1)-bit label.  Many waves
// of tiles hide the match's latency and gain from its instruction count; one
// wave is latency bound and takes the ballots.  The match form also runs four
// CTAs per SM (64 registers) to hide more of that latency.
template <bool MATCH, int RB>
__device__ __forceinline__ uint32_t lanes_with_digit(uint32_t d) {
    if (MATCH) return __match_any_sync(0xffffffffu, d);
    uint32_t peers = 0xffffffffu;
#pragma unroll
    for (int b = 0; b <= RB; ++b) {
        const bool bit = (d >> b) & 1u;
        const uint32_t v = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? v : ~v;
    }
    return peers;
}

// Stable scatter of one tile by digit (one CTA per tile): ranks the keys in
// input order (lanes_with_digit + per-warp counters), places them by digit in
// shared memory and writes each digit's run to its global start from the
// scan.  FIRST: the values are the positions, generated instead of read
// (the first pass of a batch with per-lookup scales and no compaction).
template <bool FIRST, int RB, bool MATCH>
__global__ void __launch_bounds__(kSortThreads, MATCH ? 4 : 3) downsweep_kernel(const uint32_t* __restrict__ keys_in,
                                                                    const uint32_t* __restrict__ vals_in,
                                                                    uint32_t* __restrict__ keys_out,
                                                                    uint32_t* __restrict__ vals_out,
                                                                    const uint32_t* __restrict__ tstart_g,
                                                                    uint32_t tiles, uint32_t N,
                                                                    const uint32_t* __restrict__ nsp, int shift) {
    chain_wait();

    constexpr int RADIX = 1 << RB;
    constexpr int DPT = RADIX / kSortThreads;  // digits per thread (consecutive)
    static_assert(DPT >= 1 && DPT * kSortThreads == RADIX, "digits must split evenly over the threads");
    __shared__ uint32_t s_keys[kSortTile];
    __shared__ uint32_t s_src[kSortTile];  // tile-local source index of each sorted slot
    // per-warp digit counts, then warp-exclusive offsets (at most kSortTile: 16 bits)
    __shared__ uint16_t s_whist[kSortThreads / 32][RADIX];
    __shared__ uint32_t s_tile_start[RADIX];
    __shared__ uint32_t s_global[RADIX];
    __shared__ uint32_t s_scan[8];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d0 = tid * DPT;  // this thread's digits
    const uint32_t tile = blockIdx.x;
    const uint32_t base = tile * kSortTile;
    if (nsp) N = tmin<uint32_t>(*nsp, N);  // sorted keys (device count)
    if (base >= N) return;                 // whole CTA: a tile past the sorted keys
    for (int i = tid; i < (kSortThreads / 32) * RADIX; i += kSortThreads) (&s_whist[0][0])[i] = 0;
    // global start of this thread's digits from this tile (used after ranking)
    uint32_t gstart[DPT];
#pragma unroll
    for (int i = 0; i < DPT; ++i) gstart[i] = __ldg(tstart_g + (size_t)(d0 + i) * tiles + tile);
    __syncthreads();

    // ranks inside the warp are below 512: two per register
    uint32_t key[kSortItems], rank2[kSortItems / 2];
    const uint32_t wbase = base + warp * (32 * kSortItems) + lane;
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const uint32_t idx = wbase + k * 32;
        key[k] = idx < N ? keys_in[idx] : 0u;
    }
    // digit of item k (RADIX past the end: not ranked)
    auto digit_of = [&](int k) -> int {
        return wbase + k * 32 < N ? (int)((key[k] >> shift) & (RADIX - 1)) : RADIX;
    };
    // stable rank inside the warp, in input order (item-major, then lane)
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const int d = digit_of(k);
        const uint32_t peers = lanes_with_digit<MATCH, RB>((uint32_t)d);
        uint32_t cnt = 0;
        if (d < RADIX) cnt = s_whist[warp][d];
        const uint32_t r = cnt + __popc(peers & lt_mask);
        if (k & 1)
            rank2[k >> 1] |= r << 16;
        else
            rank2[k >> 1] = r;
        __syncwarp();
        if (d < RADIX && (peers & lt_mask) == 0) s_whist[warp][d] = (uint16_t)(cnt + __popc(peers));
        __syncwarp();
    }
    __syncthreads();
    // per digit: warp-exclusive offsets, tile total, tile-local start
    uint32_t total[DPT];
    uint32_t tsum = 0;
#pragma unroll
    for (int i = 0; i < DPT; ++i) {
        total[i] = 0;
#pragma unroll
        for (int w = 0; w < kSortThreads / 32; ++w) {
            const uint32_t c = s_whist[w][d0 + i];
            s_whist[w][d0 + i] = (uint16_t)total[i];
            total[i] += c;
        }
        tsum += total[i];
    }
    {
        uint32_t tile_total;
        uint32_t ts = block_exclusive_scan_256(tsum, s_scan, &tile_total);
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
            s_tile_start[d0 + i] = ts;
            s_global[d0 + i] = gstart[i] - ts;
            ts += total[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const int d = digit_of(k);
        if (d < RADIX) {
            const uint32_t lp = s_tile_start[d] + s_whist[warp][d] + ((rank2[k >> 1] >> (16 * (k & 1))) & 0xffffu);
            s_keys[lp] = key[k];
            s_src[lp] = wbase + k * 32 - base;
        }
    }
    __syncthreads();
    // write out in sorted order (each digit's run is contiguous); the value
    // gathers of all the thread's items are issued before any store
    const uint32_t nvalid = min((uint32_t)kSortTile, N - base);
    uint32_t vv[kSortItems];
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const uint32_t i = (uint32_t)(k * kSortThreads + tid);
        const uint32_t src = i < nvalid ? base + s_src[i] : 0u;
        vv[k] = FIRST ? src : (i < nvalid ? __ldg(vals_in + src) : 0u);
    }
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const uint32_t i = (uint32_t)(k * kSortThreads + tid);
        if (i < nvalid) {
            const uint32_t kk = s_keys[i];
            const uint32_t g = s_global[(kk >> shift) & (RADIX - 1)] + i;
            if (g < N) {
                keys_out[g] = kk;
                vals_out[g] = vv[k];
            }
        }
    }
}

// --------------------------------------------------------- run-length code

// Table of a key: the last table whose row base is <= key, or T for the key
// of skipped lookups (>= the sum of all rows).
__device__ __forceinline__ int key_table(const PrepArgs& a, uint32_t key) {
    if (key >= a.total_rows) return a.T;
    int lo = 0, hi = a.T - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((uint64_t)a.tabs[mid].rowbase <= key)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// First key past table t's key range (all keys for the skipped-lookup key T).
__device__ __forceinline__ uint32_t table_end(const PrepArgs& a, int t) {
    return t >= a.T ? 0xffffffffu : (t + 1 < a.T ? (uint32_t)a.tabs[t + 1].rowbase : a.total_rows);
}

// Run-length encoding of the sorted keys, tile by tile with a warp-parallel
// look-back for the running count of distinct keys: uniq/runstart and
// ustart[t], the first distinct-key index of every table (keys are sorted and
// each table owns a consecutive key range), ustart[T] the end.
// A thread's kSortItems consecutive sorted keys (from p0) and their head
// flags (bit q: position p0+q starts a run).
__device__ __forceinline__ uint32_t rle_load_heads(const uint32_t* __restrict__ skeys, uint32_t N, uint32_t p0,
                                                   uint32_t (&k)[kSortItems], uint32_t& prev) {
    if (p0 + kSortItems <= N) {
        const uint4* src = reinterpret_cast<const uint4*>(skeys + p0);
#pragma unroll
        for (int q = 0; q < kSortItems / 4; ++q) {
            const uint4 v = src[q];
            k[4 * q] = v.x;
            k[4 * q + 1] = v.y;
            k[4 * q + 2] = v.z;
            k[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < kSortItems; ++q) k[q] = p0 + q < N ? skeys[p0 + q] : 0u;
    }
    prev = (p0 > 0 && p0 - 1 < N) ? skeys[p0 - 1] : 0u;
    uint32_t heads = 0;
#pragma unroll
    for (int q = 0; q < kSortItems; ++q) {
        const uint32_t p = p0 + q;
        const uint32_t before = q == 0 ? prev : k[q - 1];
        const bool h = p < N && (p == 0 || k[q] != before);
        heads |= (uint32_t)h << q;
    }
    return heads;
}

// Number of runs starting in each tile of sorted keys (one CTA per tile).
__global__ void __launch_bounds__(kSortThreads) rle_count_kernel(const uint32_t* __restrict__ skeys, uint32_t N,
                                                                 const uint32_t* __restrict__ nsp,
                                                                 uint32_t* __restrict__ tcount) {
    chain_wait();

    __shared__ uint32_t s_scan[8];
    if (nsp) N = tmin<uint32_t>(*nsp, N);  // sorted keys (device count)
    uint32_t k[kSortItems], prev;
    const uint32_t heads = rle_load_heads(skeys, N, blockIdx.x * kSortTile + threadIdx.x * kSortItems, k, prev);
    uint32_t total;
    block_exclusive_scan_256(__popc(heads), s_scan, &total);
    if (threadIdx.x == 0) tcount[blockIdx.x] = total;
}

// Exclusive scan of n counts in place by one CTA of 1024 threads; the total
// goes to *total_out.
__global__ void __launch_bounds__(1024) tile_scan_kernel(uint32_t* __restrict__ cnt, uint32_t n,
                                                         uint32_t* __restrict__ total_out) {
    chain_wait();

    __shared__ uint32_t s_warp[32];
    const uint32_t total = block_scan_row_1024(cnt, n, 0u, s_warp);
    if (threadIdx.x == 0) *total_out = total;
}

// Run-length encoding of the sorted keys, one CTA per tile, the tile's first
// distinct-key index from the scanned run counts: uniq/runstart (runstart[U]
// = N) and ustart[t], the first distinct-key index of every table (keys are
// sorted and each table owns a consecutive key range), ustart[T] the end.
__global__ void __launch_bounds__(kSortThreads) rle_kernel(PrepArgs a, Workspace ws, const uint32_t* __restrict__ skeys) {
    chain_wait();

    __shared__ uint32_t s_scan[8];
    const uint32_t N = sorted_count(a, ws);
    const int tid = threadIdx.x;
    const uint32_t tile = blockIdx.x;
    if (N == 0) {  // every lookup belongs to a dense table: no runs
        if (tile == 0) {
            for (int t = tid; t <= a.T; t += blockDim.x) ws.ustart[t] = 0;
            if (tid == 0) ws.runstart[0] = 0;
        }
        return;
    }
    const uint32_t p0 = tile * kSortTile + tid * kSortItems;
    uint32_t k[kSortItems], prev;
    const uint32_t heads = rle_load_heads(skeys, N, p0, k, prev);
    uint32_t tile_total;
    const uint32_t excl = block_exclusive_scan_256(__popc(heads), s_scan, &tile_total);
    const uint32_t U = tmin<uint32_t>(ws.counters[CTR_U], N);
    uint32_t u = ws.tcount[tile] + excl;
    // the table of the previous key, kept with the end of its key range:
    // sorted neighbours mostly share a table, so the search runs about once
    // per table change
    int tprev = -1;
    uint32_t t_hi = 0u;  // first key past tprev's range
    if (p0 > 0 && p0 <= N) {
        tprev = key_table(a, prev);
        t_hi = table_end(a, tprev);
    }
#pragma unroll
    for (int q = 0; q < kSortItems; ++q) {
        if (!(heads & (1u << q))) continue;
        const uint32_t p = p0 + q, key = k[q];
        if (u < N) {
            ws.uniq[u] = key;
            ws.runstart[u] = p;
            // tables whose key range starts after the previous key and at or
            // before this one begin at u
            if (tprev < 0 || key >= t_hi) {
                const int tk = key_table(a, key);
                for (int t2 = tprev + 1; t2 <= tk; ++t2) ws.ustart[t2] = u;
                tprev = tk;
                t_hi = table_end(a, tk);
            }
        }
        ++u;
    }
    // the thread holding the last position ends the table ranges
    if (N > 0 && p0 <= N - 1 && N - 1 < p0 + kSortItems) {
        const int tlast = key_table(a, skeys[N - 1]);
        for (int t2 = tlast + 1; t2 <= a.T; ++t2) ws.ustart[t2] = U;
        ws.runstart[U] = N;
    }
}

// Chunks of the long runs, numbered in key order after the run-length
// encoding (count, scan, write over tiles of kSortTile distinct keys): every
// run of at least kLongRun lookups gets its first chunk g0, the number of
// chunks of all earlier runs; the run's ceil(len / chunk) chunks g0 ..
// get (u, g0) and the run's finished-chunk count (kept at g0) is cleared.
// cstart[t] is the first chunk of table t (the chunk base at its first
// distinct key) and cstart[T] the total, so the chunks of each table are one
// consecutive range in key order.

// Chunk counts of the runs of a thread's kSortItems distinct keys from u0.
__device__ __forceinline__ void run_chunks(const PrepArgs& a, const Workspace& ws, uint32_t U, uint32_t u0,
                                           uint32_t (&nc)[kSortItems]) {
    const uint32_t N = sorted_count(a, ws);
    uint32_t rs[kSortItems + 1];
    if (u0 + kSortItems <= U) {
        const uint4* src = reinterpret_cast<const uint4*>(ws.runstart + u0);
#pragma unroll
        for (int q = 0; q < kSortItems / 4; ++q) {
            const uint4 v = src[q];
            rs[4 * q] = v.x;
            rs[4 * q + 1] = v.y;
            rs[4 * q + 2] = v.z;
            rs[4 * q + 3] = v.w;
        }
        rs[kSortItems] = u0 + kSortItems < U ? ws.runstart[u0 + kSortItems] : N;
    } else {
#pragma unroll
        for (int q = 0; q <= kSortItems; ++q) rs[q] = u0 + q < U ? ws.runstart[u0 + q] : N;
    }
#pragma unroll
    for (int q = 0; q < kSortItems; ++q) {
        nc[q] = 0;
        const uint32_t r0 = tmin<uint32_t>(rs[q], N), r1 = tmin<uint32_t>(rs[q + 1], N);
        if (u0 + q < U && r1 > r0 && r1 - r0 >= (uint32_t)kLongRun && ws.uniq[u0 + q] < a.total_rows)
            nc[q] = (r1 - r0 + (uint32_t)a.chunk - 1) / (uint32_t)a.chunk;
    }
}

// Chunks per tile of distinct keys (tiles past the distinct keys count 0).
__global__ void __launch_bounds__(kSortThreads) chunk_count_kernel(PrepArgs a, Workspace ws, uint32_t tiles) {
    chain_wait();

    __shared__ uint32_t s_scan[8];
    const uint32_t U = tmin<uint32_t>(ws.counters[CTR_U], (uint32_t)a.N);
    for (uint32_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        if (tile * kSortTile >= U) {
            if (threadIdx.x == 0) ws.tcount[tile] = 0;
            continue;
        }
        uint32_t nc[kSortItems], sum = 0;
        run_chunks(a, ws, U, tile * kSortTile + threadIdx.x * kSortItems, nc);
#pragma unroll
        for (int q = 0; q < kSortItems; ++q) sum += nc[q];
        uint32_t total;
        block_exclusive_scan_256(sum, s_scan, &total);
        if (threadIdx.x == 0) ws.tcount[tile] = total;
    }
}

// The chunk records and cstart, from the scanned chunk counts.
__global__ void __launch_bounds__(kSortThreads) chunk_write_kernel(PrepArgs a, Workspace ws, uint32_t tiles) {
    chain_wait();

    __shared__ uint32_t s_scan[8];
    __shared__ uint32_t s_base[kSortTile];  // exclusive chunk base of each distinct key of the tile
    const uint32_t U = tmin<uint32_t>(ws.counters[CTR_U], (uint32_t)a.N);
    const uint32_t total = tmin<uint32_t>(ws.counters[CTR_NCHUNK], (uint32_t)ws.max_chunks);
    const int tid = threadIdx.x;
    if (blockIdx.x == 0)  // tables that start at or after the last distinct key
        for (int t = tid; t <= a.T; t += blockDim.x)
            if (tmin<uint32_t>(ws.ustart[t], U) == U) ws.cstart[t] = total;
    for (uint32_t tile = blockIdx.x; tile < tiles && tile * kSortTile < U; tile += gridDim.x) {
        const uint32_t t0 = tile * kSortTile;
        const uint32_t u0 = t0 + tid * kSortItems;
        uint32_t nc[kSortItems], sum = 0;
        run_chunks(a, ws, U, u0, nc);
#pragma unroll
        for (int q = 0; q < kSortItems; ++q) sum += nc[q];
        uint32_t tile_total;
        const uint32_t excl = block_exclusive_scan_256(sum, s_scan, &tile_total);
        uint32_t base = ws.tcount[tile] + excl;
#pragma unroll
        for (int q = 0; q < kSortItems; ++q) {
            s_base[tid * kSortItems + q] = base;
            if (nc[q] && (int64_t)base + nc[q] <= ws.max_chunks) {
                for (uint32_t j = 0; j < nc[q]; ++j) ws.chunk_info[base + j] = make_uint2(u0 + q, base);
                ws.chunk_done[base] = 0;
            }
            base += nc[q];
        }
        __syncthreads();
        // first chunk of every table whose first distinct key is in this tile
        for (int t = tid; t <= a.T; t += blockDim.x) {
            const uint32_t us = tmin<uint32_t>(ws.ustart[t], U);
            if (us >= t0 && us < tmin<uint32_t>(t0 + kSortTile, U)) ws.cstart[t] = s_base[us - t0];
        }
        __syncthreads();  // s_base is reused by the next tile
    }
}

// One downsweep pass: positions generated (first pass) or read, ranking by
// warp match or by ballots.
template <int RB>
static void launch_downsweep(bool first, bool match, int tiles, cudaStream_t s, const uint32_t* kin,
                             const uint32_t* vin, uint32_t* kout, uint32_t* vout, const uint32_t* tstart,
                             uint32_t nt, uint32_t n, const uint32_t* nsp, int shift) {
    auto* k = first ? (match ? downsweep_kernel<true, RB, true> : downsweep_kernel<true, RB, false>)
                    : (match ? downsweep_kernel<false, RB, true> : downsweep_kernel<false, RB, false>);
    launch_chained(k, dim3(tiles), dim3(kSortThreads), s, kin, vin, kout, vout, tstart, nt, n, nsp, shift);
}

// One wave of keys_kernel CTAs (three per SM).
template <typename IDX>
static cudaError_t launch_keys(const PrepArgs& a, Workspace& ws, int64_t tiles, int sms, cudaStream_t s) {
    const unsigned grid = (unsigned)tmin<int64_t>(tiles, (int64_t)sms * 3);
    return launch_chained(keys_kernel<IDX>, dim3(grid), dim3(256), s, a, ws);
}

// ------------------------------------------------------------------ launch

cudaError_t launch_prepare(const PrepArgs& a, Workspace& ws, cudaStream_t s) {
    if (a.N == 0) {
        ws.sorted_buf = 0;
        return cudaMemsetAsync(ws.ustart, 0, sizeof(uint32_t) * (a.T + 1), s);
    }
    const int tiles = (int)((a.N + kSortTile - 1) / kSortTile);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t nbags = (int64_t)a.T * a.B;
    const unsigned mgrid = (unsigned)tmax<int64_t>(1, tmin<int64_t>((nbags + 256) / 256, (int64_t)sms * 8));
    cudaError_t e;
    if (a.idx64)
        bag_marks_kernel<int64_t><<<mgrid, 256, 0, s>>>(a, ws);
    else
        bag_marks_kernel<int32_t><<<mgrid, 256, 0, s>>>(a, ws);
    // dense tables present: only the other tables' keys are sorted, compacted
    if (a.compact) launch_chained(compact_kernel, dim3(1), dim3(1024), s, a, ws);
    e = a.idx64 ? launch_keys<int64_t>(a, ws, tiles, sms, s) : launch_keys<int32_t>(a, ws, tiles, sms, s);
    if (e != cudaSuccess) return e;
    const uint32_t* nsp = a.compact ? ws.counters + CTR_NS : nullptr;  // sorted keys (device count)
    // upsweep CTAs: each walks several tiles when there are more than four
    // CTAs' worth per SM, so fewer partial histograms meet in global atomics
    const unsigned ugrid = (unsigned)tmin<int64_t>(tiles, (int64_t)sms * 4);
    // downsweep ranking: warp match beyond one wave of tiles (3 CTAs per SM)
    const bool match = tiles > sms * 3;
    int cur = 0;
    for (int p = 0; p < ws.passes; ++p) {
        // the first pass numbers the positions itself unless the keys kernel
        // wrote the values (compacted keys, or bags when there is no scale);
        // the keys kernel counted the first pass's digits unless compacted
        const bool counted = p == 0 && !a.compact;
        const bool gen = counted && ws.scale != nullptr;
        const uint32_t* kin = ws.keys[cur];
        const uint32_t* vin = gen ? nullptr : ws.vals[cur];
        uint32_t* kout = ws.keys[cur ^ 1];
        uint32_t* vout = ws.vals[cur ^ 1];
        uint32_t* hp = ws.hist + p * kMaxRadix;
        const int shift = p * ws.digit_bits;
        const uint32_t nt = (uint32_t)tiles, n = (uint32_t)a.N;
        if (ws.digit_bits == 9) {
            if (!counted) launch_chained(upsweep_kernel<9>, dim3(ugrid), dim3(kSortThreads), s, kin, n, nsp, shift, ws.tcount, nt, hp);
            launch_scan<9>(ws.tcount, hp, nt, n, nsp, s);
            launch_downsweep<9>(gen, match, tiles, s, kin, vin, kout, vout, ws.tcount, nt, n, nsp, shift);
        } else {
            if (!counted) launch_chained(upsweep_kernel<8>, dim3(ugrid), dim3(kSortThreads), s, kin, n, nsp, shift, ws.tcount, nt, hp);
            launch_scan<8>(ws.tcount, hp, nt, n, nsp, s);
            launch_downsweep<8>(gen, match, tiles, s, kin, vin, kout, vout, ws.tcount, nt, n, nsp, shift);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        cur ^= 1;
    }
    ws.sorted_buf = cur;
    launch_chained(rle_count_kernel, dim3(tiles), dim3(kSortThreads), s, (const uint32_t*)ws.keys[cur], (uint32_t)a.N, nsp, ws.tcount);
    launch_chained(tile_scan_kernel, dim3(1), dim3(1024), s, ws.tcount, (uint32_t)tiles, ws.counters + CTR_U);
    launch_chained(rle_kernel, dim3(tiles), dim3(kSortThreads), s, a, ws, (const uint32_t*)ws.keys[cur]);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned cgrid = (unsigned)tmin<int64_t>(tiles, (int64_t)sms * 4);
    launch_chained(chunk_count_kernel, dim3(cgrid), dim3(kSortThreads), s, a, ws, (uint32_t)tiles);
    launch_chained(tile_scan_kernel, dim3(1), dim3(1024), s, ws.tcount, (uint32_t)tiles, ws.counters + CTR_NCHUNK);
    launch_chained(chunk_write_kernel, dim3(cgrid), dim3(kSortThreads), s, a, ws, (uint32_t)tiles);
    return cudaGetLastError();
}

}  // namespace tbe
