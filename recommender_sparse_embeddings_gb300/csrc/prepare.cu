// Backward preparation: transpose, sort, run-length encoding (kimbodo
// "Kimbodo Engineering Perspective" names these three steps; kimbodo "What
// Happened": updates are grouped by (table, row)).
//
//  1. keys_kernel: one (table,row) key per lookup, key = rowbase_t + idx (or
//     the sentinel sum-of-rows for an index out of range), the flat bag of
//     each position, the lookup's scale s_i when weights or mean pooling
//     apply, and the digit histograms of every radix pass.  Positions are
//     tiled evenly, so bag lengths do not unbalance the work.
//  2. onesweep_kernel, once per 8-bit digit: a stable LSD radix pass.  Each
//     CTA claims the next tile, ranks its keys by digit (warp match + per-warp
//     counters, in input order), learns the counts of all earlier tiles by a
//     bounded decoupled look-back, and scatters through shared memory so each
//     digit's run is written contiguously.  The first pass generates the
//     values (positions) instead of reading them.
//  3. rle_kernel: head flags of the sorted keys, a tile scan with look-back,
//     the distinct keys with their first sorted slot (runstart[U] = N), the
//     registration of long runs and the first distinct key of each table.
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

template <typename IDX>
__global__ void __launch_bounds__(256) keys_kernel(PrepArgs a, Workspace ws) {
    __shared__ int64_t s_off[kKeysWindow];
    __shared__ uint32_t s_hist[kMaxPasses][kRadix];
    __shared__ int64_t s_first, s_last;
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const int64_t nbags = (int64_t)a.T * a.B;
    const int passes = (a.key_bits + kRadixBits - 1) / kRadixBits;
    uint32_t err = 0;

    for (int i = threadIdx.x; i < kMaxPasses * kRadix; i += blockDim.x) (&s_hist[0][0])[i] = 0;

    // offsets check, grid-stride over bags
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g <= nbags;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = ld_index(off, g);
        if (o < 0 || o > a.N) err |= ERR_OFFSETS;
        if (g == 0 && o != 0) err |= ERR_OFFSETS;
        if (g == nbags && o != a.N) err |= ERR_OFFSETS;
        if (g < nbags && ld_index(off, g + 1) < o) err |= ERR_OFFSETS;
    }

    const int64_t tiles = (a.N + kSortTile - 1) / kSortTile;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t p0 = tile * kSortTile;
        const int64_t p1 = min(p0 + (int64_t)kSortTile, a.N);
        __syncthreads();
        {
            const int64_t f = block_find_bag(off, nbags, p0);
            const int64_t l = block_find_bag(off, nbags, p1 - 1);
            if (threadIdx.x == 0) {
                s_first = f;
                s_last = l;
            }
        }
        __syncthreads();
        const int64_t bf = s_first, bl = min(s_last, nbags - 1);
        const int64_t nwin = bl - bf + 2;  // offsets bf .. bl+1
        const bool staged = nwin <= kKeysWindow && bl >= bf;
        if (staged)
            for (int64_t k = threadIdx.x; k < nwin; k += blockDim.x) s_off[k] = ld_index(off, bf + k);
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kSortItems; ++k) {
            const int64_t p = p0 + (int64_t)k * blockDim.x + threadIdx.x;
            if (p >= p1) continue;
            int64_t bag, bstart, bend;
            if (staged) {
                int64_t lo = 0, hi = nwin;  // first window slot with offset > p
                while (lo < hi) {
                    const int64_t mid = (lo + hi) >> 1;
                    if (s_off[mid] > p)
                        hi = mid;
                    else
                        lo = mid + 1;
                }
                const int64_t j = tmax<int64_t>(tmin<int64_t>(lo - 1, nwin - 2), 0);
                bag = bf + j;
                bstart = s_off[j];
                bend = s_off[j + 1];
            } else {
                bag = upper_bound_global(off, bf, min(bl + 2, nbags + 1), p) - 1;
                bag = tmax<int64_t>(tmin<int64_t>(bag, nbags - 1), 0);
                bstart = ld_index(off, bag);
                bend = ld_index(off, bag + 1);
            }
            const int t = (int)(bag / a.B);
            const int64_t rows = a.tabs[t].rows;
            const int64_t x = ld_index(ind, p);
            uint32_t key = a.total_rows;
            if (x >= 0 && x < rows)
                key = (uint32_t)(a.tabs[t].rowbase + x);
            else
                err |= ERR_OOB;
            ws.keys[0][p] = key;
            ws.bag[p] = (uint32_t)bag;
            if (ws.scale) {
                float s = a.weights ? __ldg(a.weights + p) : 1.f;
                const int64_t L = bend - bstart;
                if (a.mean && L > 0) s = __fdiv_rn(s, (float)L);
                ws.scale[p] = s;
            }
            for (int q = 0; q < passes; ++q) atomicAdd(&s_hist[q][(key >> (q * kRadixBits)) & (kRadix - 1)], 1u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x) {
        const uint32_t c = (&s_hist[0][0])[i];
        if (c) atomicAdd(ws.hist + i, c);
    }
    if (err) atomicOr(&a.blk->error, err);
}

// --------------------------------------------------------- one radix pass

template <bool FIRST>
__global__ void __launch_bounds__(kSortThreads) onesweep_kernel(const uint32_t* __restrict__ keys_in,
                                                                const uint32_t* __restrict__ vals_in,
                                                                uint32_t* __restrict__ keys_out,
                                                                uint32_t* __restrict__ vals_out,
                                                                const uint32_t* __restrict__ hist,
                                                                uint32_t* status, uint32_t* tile_ctr,
                                                                uint32_t N, int shift, uint32_t* err) {
    __shared__ uint32_t s_keys[kSortTile];
    __shared__ uint32_t s_vals[kSortTile];
    __shared__ uint32_t s_whist[kSortThreads / 32][kRadix];
    __shared__ uint32_t s_tile_start[kRadix];
    __shared__ uint32_t s_global[kRadix];
    __shared__ uint32_t s_scan[8];
    __shared__ uint32_t s_tile;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_tile = atomicAdd(tile_ctr, 1u);
    for (int i = tid; i < (kSortThreads / 32) * kRadix; i += kSortThreads) (&s_whist[0][0])[i] = 0;
    // global start of each digit bin
    uint32_t tot;
    const uint32_t bin_start = block_exclusive_scan_256(hist[tid], s_scan, &tot);
    __syncthreads();
    const int tile = (int)s_tile;
    const uint32_t base = (uint32_t)tile * kSortTile;

    uint32_t key[kSortItems], val[kSortItems], rank[kSortItems];
    int digit[kSortItems];
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const uint32_t idx = base + warp * (32 * kSortItems) + k * 32 + lane;
        if (idx < N) {
            key[k] = keys_in[idx];
            val[k] = FIRST ? idx : vals_in[idx];
            digit[k] = (key[k] >> shift) & (kRadix - 1);
        } else {
            key[k] = 0;
            val[k] = 0;
            digit[k] = kRadix;  // past the end: not ranked
        }
    }
    // stable rank inside the warp, in input order (item-major, then lane)
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const int d = digit[k];
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        uint32_t cnt = 0;
        if (d < kRadix) cnt = s_whist[warp][d];
        rank[k] = cnt + __popc(peers & lt_mask);
        __syncwarp();
        if (d < kRadix && (peers & lt_mask) == 0) s_whist[warp][d] = cnt + __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // per digit: warp-exclusive offsets, tile total, look-back, tile-local start
    uint32_t total = 0;
#pragma unroll
    for (int w = 0; w < kSortThreads / 32; ++w) {
        const uint32_t c = s_whist[w][tid];
        s_whist[w][tid] = total;
        total += c;
    }
    const uint32_t prefix = lookback(status + tid, tile, kRadix, total, err);
    uint32_t tile_total;
    const uint32_t tstart = block_exclusive_scan_256(total, s_scan, &tile_total);
    s_tile_start[tid] = tstart;
    s_global[tid] = bin_start + prefix - tstart;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kSortItems; ++k) {
        const int d = digit[k];
        if (d < kRadix) {
            const uint32_t lp = s_tile_start[d] + s_whist[warp][d] + rank[k];
            s_keys[lp] = key[k];
            s_vals[lp] = val[k];
        }
    }
    __syncthreads();
    const uint32_t nvalid = min((uint32_t)kSortTile, N - base);
    for (uint32_t i = tid; i < nvalid; i += kSortThreads) {
        const uint32_t k = s_keys[i];
        const uint32_t g = s_global[(k >> shift) & (kRadix - 1)] + i;
        if (g < N) {
            keys_out[g] = k;
            vals_out[g] = s_vals[i];
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
// look-back for the running count of distinct keys.  Besides uniq/runstart
// it does the two jobs the apply step needs from the run boundaries:
//  - registers every run of at least kLongRun lookups for the accumulate
//    path (a run starting at p is long iff the key at p + 255 equals the key
//    at p; its end is then found by an exponential then binary search):
//    ceil(len / kLongRun) consecutive chunk slots and a record (unique index,
//    first chunk, chunk count, chunks finished = 0);
//  - ustart[t]: the first distinct-key index of every table (keys are sorted
//    and each table owns a consecutive key range), ustart[T] the end.
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
            // long run: registered for the accumulate path
            if (key < a.total_rows && p + (kLongRun - 1) < N && __ldg(skeys + p + kLongRun - 1) == key) {
                uint32_t lo = p + kLongRun - 1, step = kLongRun;  // skeys[lo] == key
                while (lo + step < N && __ldg(skeys + lo + step) == key) {
                    lo += step;
                    step *= 2;
                }
                uint32_t hi = tmin<uint32_t>(lo + step, N);  // first differing slot is in (lo, hi]
                while (hi - lo > 1) {
                    const uint32_t mid = lo + (hi - lo) / 2;
                    if (__ldg(skeys + mid) == key)
                        lo = mid;
                    else
                        hi = mid;
                }
                const uint32_t len = hi - p;
                const uint32_t nc = (len + kLongRun - 1) / kLongRun;
                const uint32_t base = atomicAdd(&ws.counters[CTR_NCHUNK], nc);
                const uint32_t li = atomicAdd(&ws.counters[CTR_NLONG], 1u);
                if (li < ws.max_long && (int64_t)base + nc <= ws.max_chunks) {
                    ws.long_runs[4 * li + 0] = u;
                    ws.long_runs[4 * li + 1] = base;
                    ws.long_runs[4 * li + 2] = nc;
                    ws.long_runs[4 * li + 3] = 0;
                    // the chunks join the list of the table's backward class
                    // (at most the registered total, so within max_chunks)
                    const int slot = a.tabs[tk].cslot;
                    const uint32_t lc = atomicAdd(&ws.counters[CTR_CLS_CHUNK + slot], nc);
                    uint2* list = ws.cls_chunks + (int64_t)slot * ws.max_chunks + lc;
                    for (uint32_t j = 0; j < nc; ++j) list[j] = make_uint2(li, j);
                }
            }
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
    const unsigned kgrid = (unsigned)min(tiles, sms * 4);
    if (a.idx64)
        keys_kernel<int64_t><<<kgrid, 256, 0, s>>>(a, ws);
    else
        keys_kernel<int32_t><<<kgrid, 256, 0, s>>>(a, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int cur = 0;
    for (int p = 0; p < ws.passes; ++p) {
        uint32_t* st = ws.status + (size_t)p * tiles * kRadix;
        uint32_t* ctr = ws.counters + CTR_PASS_TILE + p;
        if (p == 0)
            onesweep_kernel<true><<<tiles, kSortThreads, 0, s>>>(ws.keys[cur], nullptr, ws.keys[cur ^ 1],
                                                                 ws.vals[cur ^ 1], ws.hist + p * kRadix, st, ctr,
                                                                 (uint32_t)a.N, p * kRadixBits, &a.blk->error);
        else
            onesweep_kernel<false><<<tiles, kSortThreads, 0, s>>>(ws.keys[cur], ws.vals[cur], ws.keys[cur ^ 1],
                                                                  ws.vals[cur ^ 1], ws.hist + p * kRadix, st, ctr,
                                                                  (uint32_t)a.N, p * kRadixBits, &a.blk->error);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        cur ^= 1;
    }
    ws.sorted_buf = cur;
    rle_kernel<<<tiles, kSortThreads, 0, s>>>(a, ws, ws.keys[cur]);
    return cudaGetLastError();
}

}  // namespace tbe
