// Backward preparation: transpose, sort, run-length encoding (kimbodo
// "Kimbodo Engineering Perspective" names these three steps; kimbodo "What
// Happened": updates are grouped by (table, row)).
//
//  1. bag_marks_kernel + keys_kernel: one (table,row) key per lookup, key =
//     rowbase_t + idx (or the sentinel sum-of-rows for an index out of
//     range), the flat bag of each position, the lookup's scale s_i when
//     weights or mean pooling apply, and the digit histograms of every radix
//     pass.  Positions are tiled evenly (the first bag of each tile is marked
//     by a pass over the bags), so bag lengths do not unbalance the work.
//  2. onesweep_kernel, once per 8-bit digit: a stable LSD radix pass.  Each
//     CTA claims the next tile, ranks its keys by digit (warp match + per-warp
//     counters, in input order), learns the counts of all earlier tiles by a
//     bounded decoupled look-back, and scatters through shared memory so each
//     digit's run is written contiguously.  The first pass generates the
//     values (positions) instead of reading them.
//  3. rle_kernel: head flags of the sorted keys, a tile scan with look-back,
//     the distinct keys with their first sorted slot (runstart[U] = N) and
//     the first distinct key of each table.
//  4. chunk_scan_kernel: numbers the 256-lookup chunks of every run of at
//     least kLongRun lookups in key order (a scan over the distinct keys), so
//     each table's chunks form one consecutive range for the apply step.
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

// Offsets check and the first bag of every key tile: a grid-stride pass over
// the bags; a bag [o, o1) marks every tile whose first position it holds, so
// with valid offsets each tile start is marked exactly once (by the bag that
// contains it).  Malformed offsets leave some marks stale or zero; the keys
// kernel only uses marks to narrow its search and stays in range regardless.
template <typename IDX>
__global__ void __launch_bounds__(256) bag_marks_kernel(PrepArgs a, Workspace ws) {
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const int64_t nbags = (int64_t)a.T * a.B;
    uint32_t err = 0;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g <= nbags;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = ld_index(off, g);
        if (o < 0 || o > a.N) err |= ERR_OFFSETS;
        if (g == 0 && o != 0) err |= ERR_OFFSETS;
        if (g == nbags && o != a.N) err |= ERR_OFFSETS;
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

// Asynchronous global -> shared copy of one element (4 or 8 bytes), and the
// wait for all of a thread's copies.
template <int BYTES>
__device__ __forceinline__ void cp_async(void* smem, const void* gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(gmem), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Dynamic shared memory of keys_kernel: the tile's indices and weights
// (copied asynchronously while the bag map is built), the staged offsets and
// the bag marks.
template <typename IDX>
constexpr size_t keys_smem_bytes(bool weights) {
    return sizeof(IDX) * kSortTile + (weights ? sizeof(float) * kSortTile : 0) + sizeof(int32_t) * (kKeysWindow + 3) +
           sizeof(int16_t) * kSortTile;
}

// One key per position, tile by tile.  The tile's indices and weights are
// copied to shared memory asynchronously first, so their DRAM latency
// overlaps the rest of the set-up.  The tile's bags [bf, bl] come from the
// marks (the last tile finds its last bag with a block-wide search); their
// offsets are staged in shared memory and every position learns its bag from
// a position -> bag map: each non-empty bag marks its first position in the
// tile, and an inclusive max-scan over the tile's positions carries each
// mark forward to the bag's last position.  Warp w takes positions
// w*512 + k*32 + lane (k < 16), so global stores are coalesced and the scan
// runs in registers with shuffles.  The digit histograms of all radix passes
// are counted per block (equal digits of a warp added once, by warp match)
// and added to the global histograms at the end.
template <typename IDX>
__global__ void __launch_bounds__(256) keys_kernel(PrepArgs a, Workspace ws) {
    extern __shared__ __align__(16) unsigned char keys_smem[];
    IDX* s_x = reinterpret_cast<IDX*>(keys_smem);
    float* s_w = reinterpret_cast<float*>(keys_smem + sizeof(IDX) * kSortTile);
    int32_t* s_off = reinterpret_cast<int32_t*>(keys_smem + sizeof(IDX) * kSortTile +
                                                (a.weights ? sizeof(float) * kSortTile : 0));
    int16_t* s_mark = reinterpret_cast<int16_t*>(s_off + kKeysWindow + 3);  // window index of the bag starting here
    __shared__ uint32_t s_hist[kMaxPasses][kMaxRadix];
    __shared__ int32_t s_wmax[kSortThreads / 32];
    __shared__ int64_t s_last;
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const int64_t nbags = (int64_t)a.T * a.B;
    const int dbits = a.digit_bits;
    const uint32_t dmask = (1u << dbits) - 1u;
    const int passes = (a.key_bits + dbits - 1) / dbits;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t Nc = a.N;  // offsets are clamped to [0, N] when staged
    uint32_t err = 0;

    for (int i = threadIdx.x; i < kMaxPasses * kMaxRadix; i += blockDim.x) (&s_hist[0][0])[i] = 0;

    const int64_t tiles = (a.N + kSortTile - 1) / kSortTile;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t p0 = tile * kSortTile;
        const int64_t p1 = min(p0 + (int64_t)kSortTile, a.N);
        const int n = (int)(p1 - p0);
        __syncthreads();  // the previous tile is done with the shared arrays
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            cp_async<sizeof(IDX)>(s_x + i, ind + p0 + i);
            if (a.weights) cp_async<4>(s_w + i, a.weights + p0 + i);
        }
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
        int bj[kSortItems];  // window index of each item's bag (staged tiles)
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
            // inclusive max-scan: per warp over its 512 positions, then across warps
            int carry = -1;
#pragma unroll
            for (int k = 0; k < kSortItems; ++k) {
                int v = s_mark[warp * (32 * kSortItems) + k * 32 + lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v = max(v, y);
                }
                v = max(v, carry);
                carry = __shfl_sync(0xffffffffu, v, 31);
                bj[k] = v;
            }
            if (lane == 0) s_wmax[warp] = carry;
        }
        cp_async_wait_all();
        __syncthreads();  // marks, warp maxima and every thread's copies are visible
        if (staged) {
            int pre = 0;  // positions before the first mark belong to bag bf (index 0)
            for (int w = 0; w < warp; ++w) pre = max(pre, s_wmax[w]);
#pragma unroll
            for (int k = 0; k < kSortItems; ++k) bj[k] = tmin<int>(max(bj[k], pre), (int)nwin - 2);
        }
        uint32_t keyv[kSortItems];
#pragma unroll
        for (int k = 0; k < kSortItems; ++k) {
            const int li = warp * (32 * kSortItems) + k * 32 + lane;
            const int64_t p = p0 + li;
            keyv[k] = 0xffffffffu;
            if (li < n) {
                int64_t bag, bstart, bend;
                if (staged) {
                    const int j = bj[k];
                    bag = bf + j;
                    bstart = s_off[j];
                    bend = s_off[j + 1];
                } else {
                    bag = upper_bound_global(off, bf, min(bl + 2, nbags + 1), p) - 1;
                    bag = tmax<int64_t>(tmin<int64_t>(bag, nbags - 1), 0);
                    bstart = ld_index(off, bag);
                    bend = ld_index(off, bag + 1);
                }
                const int t = (int)((uint32_t)bag / (uint32_t)a.B);  // T*B < 2^31
                const int64_t rows = a.tabs[t].rows;
                const int64_t x = (int64_t)s_x[li];
                uint32_t key = a.total_rows;
                if (x >= 0 && x < rows)
                    key = (uint32_t)(a.tabs[t].rowbase + x);
                else
                    err |= ERR_OOB;
                keyv[k] = key;
                ws.keys[0][p] = key;
                ws.bag[p] = (uint32_t)bag;
                if (ws.scale) {
                    float sc = a.weights ? s_w[li] : 1.f;
                    const int64_t L = bend - bstart;
                    if (a.mean && L > 0) sc = __fdiv_rn(sc, (float)L);
                    ws.scale[p] = sc;
                }
            }
        }
        // digit counts: per pass, the lowest lane of each group of equal
        // digits adds the group's size (the high digits take few values, so
        // lane-by-lane atomics would serialize on one counter)
#pragma unroll
        for (int k = 0; k < kSortItems; ++k) {
            const bool valid = warp * (32 * kSortItems) + k * 32 + lane < n;
            for (int q = 0; q < passes; ++q) {
                const uint32_t d = valid ? (keyv[k] >> (q * dbits)) & dmask : 0xffffffffu;
                const uint32_t peers = __match_any_sync(0xffffffffu, d);
                if (valid && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(&s_hist[q][d], (uint32_t)__popc(peers));
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < passes * kMaxRadix; i += blockDim.x) {
        const uint32_t c = (&s_hist[0][0])[i];
        if (c) atomicAdd(ws.hist + i, c);
    }
    if (err) atomicOr(&a.blk->error, err);
}

// One wave of keys_kernel CTAs (as many as fit per SM with this shared memory).
template <typename IDX>
static cudaError_t launch_keys(const PrepArgs& a, Workspace& ws, int64_t tiles, int sms, cudaStream_t s) {
    const bool w = a.weights != nullptr;
    const size_t smem = keys_smem_bytes<IDX>(w);
    static int per_sm[2] = {0, 0};  // resident CTAs per SM, without / with weights
    if (per_sm[w] == 0) {
        cudaError_t e = cudaFuncSetAttribute(keys_kernel<IDX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)keys_smem_bytes<IDX>(true));
        int n = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, keys_kernel<IDX>, 256, smem);
        if (e != cudaSuccess) return e;
        per_sm[w] = n > 0 ? n : 1;
    }
    const unsigned grid = (unsigned)tmin<int64_t>(tiles, (int64_t)sms * per_sm[w]);
    keys_kernel<IDX><<<grid, 256, smem, s>>>(a, ws);
    return cudaGetLastError();
}

// --------------------------------------------------------- one radix pass

template <bool FIRST, int RB>
__global__ void __launch_bounds__(kSortThreads, 3) onesweep_kernel(const uint32_t* __restrict__ keys_in,
                                                                   const uint32_t* __restrict__ vals_in,
                                                                   uint32_t* __restrict__ keys_out,
                                                                   uint32_t* __restrict__ vals_out,
                                                                   const uint32_t* __restrict__ hist,
                                                                   uint32_t* status, uint32_t* tile_ctr,
                                                                   uint32_t N, int shift, uint32_t* err) {
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
    __shared__ uint32_t s_tile;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d0 = tid * DPT;  // this thread's digits
    if (tid == 0) s_tile = atomicAdd(tile_ctr, 1u);
    for (int i = tid; i < (kSortThreads / 32) * RADIX; i += kSortThreads) (&s_whist[0][0])[i] = 0;
    // global start of each digit bin
    uint32_t bin_start[DPT];
    {
        uint32_t hsum = 0;
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
            bin_start[i] = hist[d0 + i];
            hsum += bin_start[i];
        }
        uint32_t tot;
        uint32_t ex = block_exclusive_scan_256(hsum, s_scan, &tot);
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
            const uint32_t c = bin_start[i];
            bin_start[i] = ex;
            ex += c;
        }
    }
    __syncthreads();
    const int tile = (int)s_tile;
    const uint32_t base = (uint32_t)tile * kSortTile;

    // keys in registers; values stay in memory until the final write, which
    // gathers them from this tile's input through the item's source index
    uint32_t key[kSortItems], rank[kSortItems];
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
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        uint32_t cnt = 0;
        if (d < RADIX) cnt = s_whist[warp][d];
        rank[k] = cnt + __popc(peers & lt_mask);
        __syncwarp();
        if (d < RADIX && (peers & lt_mask) == 0) s_whist[warp][d] = (uint16_t)(cnt + __popc(peers));
        __syncwarp();
    }
    __syncthreads();
    // per digit: warp-exclusive offsets, tile total, look-back, tile-local start
    uint32_t total[DPT];
#pragma unroll
    for (int i = 0; i < DPT; ++i) {
        total[i] = 0;
#pragma unroll
        for (int w = 0; w < kSortThreads / 32; ++w) {
            const uint32_t c = s_whist[w][d0 + i];
            s_whist[w][d0 + i] = (uint16_t)total[i];
            total[i] += c;
        }
    }
    uint32_t prefix[DPT];
    lookback<DPT>(status, tile, RADIX, d0, total, prefix, err);
    {
        uint32_t tsum = 0;
#pragma unroll
        for (int i = 0; i < DPT; ++i) tsum += total[i];
        uint32_t tile_total;
        uint32_t tstart = block_exclusive_scan_256(tsum, s_scan, &tile_total);
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
            s_tile_start[d0 + i] = tstart;
            s_global[d0 + i] = bin_start[i] + prefix[i] - tstart;
            tstart += total[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const int d = digit_of(k);
        if (d < RADIX) {
            const uint32_t lp = s_tile_start[d] + s_whist[warp][d] + rank[k];
            s_keys[lp] = key[k];
            s_src[lp] = wbase + k * 32 - base;
        }
    }
    __syncthreads();
    // write out in sorted order; the value gathers of all items are issued
    // together (fully unrolled) so their latencies overlap
    const uint32_t nvalid = min((uint32_t)kSortTile, N - base);
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const uint32_t i = (uint32_t)(k * kSortThreads + tid);
        if (i < nvalid) {
            const uint32_t kk = s_keys[i];
            const uint32_t src = base + s_src[i];
            const uint32_t g = s_global[(kk >> shift) & (RADIX - 1)] + i;
            if (g < N) {
                keys_out[g] = kk;
                vals_out[g] = FIRST ? src : __ldg(vals_in + src);
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

// Run-length encoding of the sorted keys, tile by tile with a warp-parallel
// look-back for the running count of distinct keys: uniq/runstart and
// ustart[t], the first distinct-key index of every table (keys are sorted and
// each table owns a consecutive key range), ustart[T] the end.
__global__ void __launch_bounds__(kSortThreads) rle_kernel(PrepArgs a, Workspace ws, const uint32_t* __restrict__ skeys) {
    __shared__ uint32_t s_scan[8];
    __shared__ uint32_t s_tile, s_prefix;
    const uint32_t N = (uint32_t)a.N;
    uint32_t* err = &a.blk->error;
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) s_tile = atomicAdd(&ws.counters[CTR_RLE_TILE], 1u);
    __syncthreads();
    const uint32_t tile = s_tile;
    const uint32_t p0 = tile * kSortTile + tid * kSortItems;
    uint32_t k[kSortItems];
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
    const uint32_t prev = (p0 > 0 && p0 - 1 < N) ? skeys[p0 - 1] : 0u;
    uint32_t heads = 0;
#pragma unroll
    for (int q = 0; q < kSortItems; ++q) {
        const uint32_t p = p0 + q;
        const uint32_t before = q == 0 ? prev : k[q - 1];
        const bool h = p < N && (p == 0 || k[q] != before);
        heads |= (uint32_t)h << q;
    }
    uint32_t tile_total;
    const uint32_t excl = block_exclusive_scan_256(__popc(heads), s_scan, &tile_total);
    if (tid < 32) {
        const uint32_t pre = lookback_warp(ws.rle_status, (int)tile, tile_total, err, lane);
        if (tid == 0) s_prefix = pre;
    }
    __syncthreads();
    const uint32_t U = tmin<uint32_t>(s_prefix + tile_total, N);
    uint32_t u = s_prefix + excl;
#pragma unroll
    for (int q = 0; q < kSortItems; ++q) {
        if (!(heads & (1u << q))) continue;
        const uint32_t p = p0 + q, key = k[q];
        if (u < N) {  // holds unless a look-back ran out (then ERR_TIMEOUT is set)
            ws.uniq[u] = key;
            ws.runstart[u] = p;
            // tables whose key range starts after the previous key and at or
            // before this one begin at u
            const int tprev = p > 0 ? key_table(a, q > 0 ? k[q - 1] : prev) : -1;
            const int tk = key_table(a, key);
            for (int t2 = tprev + 1; t2 <= tk; ++t2) ws.ustart[t2] = u;
        }
        ++u;
    }
    // the thread holding the last position ends the table ranges
    if (N > 0 && p0 <= N - 1 && N - 1 < p0 + kSortItems) {
        const int tlast = key_table(a, skeys[N - 1]);
        for (int t2 = tlast + 1; t2 <= a.T; ++t2) ws.ustart[t2] = U;
    }
    if (tid == 0 && (uint64_t)(tile + 1) * kSortTile >= N) {
        ws.counters[CTR_U] = U;
        ws.runstart[U] = N;
    }
}

// Chunks of the long runs, in key order, after the run-length kernel: a scan
// over the distinct keys (tiles of kSortTile keys claimed in order, a
// warp-parallel look-back) gives every run of at least kLongRun lookups its
// first chunk g0, the number of chunks of all earlier runs.  The run's
// ceil(len / kLongRun) chunks g0 .. get (u, g0) and the run's finished-chunk
// count (kept at g0) is cleared.  cstart[t] is the first chunk of table t
// (the chunk base at its first distinct key) and cstart[T] the total, so the
// chunks of each table are one consecutive range in key order.  Persistent
// CTAs claim tiles until the distinct keys are covered.
__global__ void __launch_bounds__(kSortThreads) chunk_scan_kernel(PrepArgs a, Workspace ws) {
    __shared__ uint32_t s_scan[8];
    __shared__ uint32_t s_base[kSortTile];  // exclusive chunk base of each distinct key of the tile
    __shared__ uint32_t s_tile, s_prefix;
    const uint32_t N = (uint32_t)a.N;
    const uint32_t U = tmin<uint32_t>(*(volatile uint32_t*)&ws.counters[CTR_U], N);
    const uint32_t utiles = (U + kSortTile - 1) / kSortTile;
    uint32_t* err = &a.blk->error;
    const int tid = threadIdx.x, lane = tid & 31;
    for (;;) {
        __syncthreads();  // the previous tile is done with the shared state
        if (tid == 0) s_tile = atomicAdd(&ws.counters[CTR_RUN_TILE], 1u);
        __syncthreads();
        const uint32_t tile = s_tile;
        if (tile >= utiles) break;
        const uint32_t t0 = tile * kSortTile;
        const uint32_t u0 = t0 + tid * kSortItems;
        // run starts u0 .. u0 + kSortItems (runstart[U] = N)
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
        uint32_t nc[kSortItems], sum = 0;
#pragma unroll
        for (int q = 0; q < kSortItems; ++q) {
            nc[q] = 0;
            const uint32_t r0 = tmin<uint32_t>(rs[q], N), r1 = tmin<uint32_t>(rs[q + 1], N);
            if (u0 + q < U && r1 > r0 && r1 - r0 >= (uint32_t)kLongRun && ws.uniq[u0 + q] < a.total_rows)
                nc[q] = (r1 - r0 + kLongRun - 1) / kLongRun;
            sum += nc[q];
        }
        uint32_t tile_total;
        const uint32_t excl = block_exclusive_scan_256(sum, s_scan, &tile_total);
        if (tid < 32) {
            const uint32_t pre = lookback_warp(ws.run_status, (int)tile, tile_total, err, lane);
            if (tid == 0) s_prefix = pre;
        }
        __syncthreads();
        uint32_t base = s_prefix + excl;
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
        const uint32_t total = s_prefix + tile_total;
        for (int t = tid; t <= a.T; t += blockDim.x) {
            const uint32_t us = tmin<uint32_t>(ws.ustart[t], U);
            if (us >= t0 && us < tmin<uint32_t>(t0 + kSortTile, U))
                ws.cstart[t] = s_base[us - t0];
            else if (us == U && tile == utiles - 1)
                ws.cstart[t] = total;
        }
        if (tid == 0 && tile == utiles - 1) ws.counters[CTR_NCHUNK] = total;
    }
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
    if (a.idx64) {
        bag_marks_kernel<int64_t><<<mgrid, 256, 0, s>>>(a, ws);
        e = launch_keys<int64_t>(a, ws, tiles, sms, s);
    } else {
        bag_marks_kernel<int32_t><<<mgrid, 256, 0, s>>>(a, ws);
        e = launch_keys<int32_t>(a, ws, tiles, sms, s);
    }
    if (e != cudaSuccess) return e;
    int cur = 0;
    const int radix = 1 << ws.digit_bits;
    for (int p = 0; p < ws.passes; ++p) {
        uint32_t* st = ws.status + (size_t)p * tiles * radix;
        uint32_t* ctr = ws.counters + CTR_PASS_TILE + p;
        const uint32_t* kin = ws.keys[cur];
        const uint32_t* vin = p == 0 ? nullptr : ws.vals[cur];
        uint32_t* kout = ws.keys[cur ^ 1];
        uint32_t* vout = ws.vals[cur ^ 1];
        const uint32_t* hp = ws.hist + p * kMaxRadix;
        const int shift = p * ws.digit_bits;
        if (ws.digit_bits == 9) {
            if (p == 0)
                onesweep_kernel<true, 9><<<tiles, kSortThreads, 0, s>>>(kin, vin, kout, vout, hp, st, ctr,
                                                                        (uint32_t)a.N, shift, &a.blk->error);
            else
                onesweep_kernel<false, 9><<<tiles, kSortThreads, 0, s>>>(kin, vin, kout, vout, hp, st, ctr,
                                                                         (uint32_t)a.N, shift, &a.blk->error);
        } else {
            if (p == 0)
                onesweep_kernel<true, 8><<<tiles, kSortThreads, 0, s>>>(kin, vin, kout, vout, hp, st, ctr,
                                                                        (uint32_t)a.N, shift, &a.blk->error);
            else
                onesweep_kernel<false, 8><<<tiles, kSortThreads, 0, s>>>(kin, vin, kout, vout, hp, st, ctr,
                                                                         (uint32_t)a.N, shift, &a.blk->error);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        cur ^= 1;
    }
    ws.sorted_buf = cur;
    rle_kernel<<<tiles, kSortThreads, 0, s>>>(a, ws, ws.keys[cur]);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned cgrid = (unsigned)tmin<int64_t>(tiles, (int64_t)sms * 2);
    chunk_scan_kernel<<<cgrid, kSortThreads, 0, s>>>(a, ws);
    return cudaGetLastError();
}

}  // namespace tbe
