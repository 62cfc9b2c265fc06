// Forward pooled lookup across all tables in one launch.
//
// What it computes ("FBTriton Rewrites Table Batched Embedding",
// "Responsibilities of the forward and backward passes"; kimbodo "What
// Happened"): out[b, Doff_t + j] = (1/L if mean) * sum_{i in bag(t,b)} s_i *
// W_t[idx_i, j], fp32 accumulation for fp32/fp16/bf16 rows.
//
// Schedule.  A row of D elements is nvec = D*elem/16 vectors of 16 bytes.  A
// "slot" of G lanes covers up to 32 vectors of a row, one vector per lane
// (G = next power of two >= nvec, at most 32).  A warp holds 32/G slots, one
// bag each; rows wider than 32 vectors are split into column blocks of 32
// vectors, each handled by its own warp.  A slot walks its bag's lookups in
// chunks: the chunk's indices and weights are loaded cooperatively
// (coalesced) one chunk ahead, then broadcast by shuffles, with U rows in
// flight per lane.  The warp -> (table, bag group, column block) map is a
// prefix over tables of ceil(B / (32/G_t)) * blocks_t warps, computed on the
// device whenever B changes.  Bags longer than kLongBag are queued for a
// second kernel where a whole CTA splits the bag into eight contiguous pieces,
// sums each with compensated (Kahan) fp32 addition, and adds the pieces in a
// fixed order.
#include "tbe_internal.cuh"

namespace tbe {

template <int DT>
struct VecTraits {
    static constexpr int E = (DT == DT_F32) ? 4 : 8;  // elements per 16-byte vector
};

// Accumulate s_i * row(idx_i) over lookups [start, end) into acc (and comp,
// the Kahan compensation, when KAHAN).  The calling slot has G lanes (mask =
// its lanes); lane `sub` owns vector vi of every row.
template <int G, int DT, typename IDX, bool KAHAN>
__device__ __forceinline__ void gather_accumulate(const uint4* __restrict__ tab, int nvec, int vi,
                                                  int64_t rows, const IDX* __restrict__ indices,
                                                  const float* __restrict__ weights, int64_t start,
                                                  int64_t end, int sub, unsigned mask,
                                                  float (&acc)[VecTraits<DT>::E],
                                                  float (&comp)[VecTraits<DT>::E], bool& oob) {
    constexpr int E = VecTraits<DT>::E;
    constexpr int J = G >= 4 ? 1 : 4 / G;  // indices held per lane per chunk
    constexpr int C = G * J;               // lookups per chunk
    constexpr int U = 4;                   // rows in flight per lane
    static_assert(C % U == 0, "chunk must split into steps");
    const bool active = vi < nvec;

    int cr[J];
    float cw[J];
    auto load_chunk = [&](int64_t c0, int(&r)[J], float(&w)[J]) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int64_t p = c0 + sub + (int64_t)j * G;
            r[j] = -1;
            w[j] = 1.f;
            if (p < end) {
                const int64_t x = ld_index(indices, p);
                if (x >= 0 && x < rows)
                    r[j] = (int)x;
                else
                    oob = true;
                if (weights) w[j] = __ldg(weights + p);
            }
        }
    };

    load_chunk(start, cr, cw);
    for (int64_t c0 = start; c0 < end; c0 += C) {
        int nr[J];
        float nw[J];
        load_chunk(c0 + C, nr, nw);  // next chunk's indices in flight with this chunk's rows
        const int n = (int)tmin<int64_t>((int64_t)C, end - c0);
#pragma unroll
        for (int k0 = 0; k0 < C; k0 += U) {
            if (k0 < n) {
                int r[U];
                float w[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    r[u] = __shfl_sync(mask, cr[(k0 + u) / G], (k0 + u) % G, G);
                    w[u] = __shfl_sync(mask, cw[(k0 + u) / G], (k0 + u) % G, G);
                }
                uint4 x[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    x[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (r[u] >= 0 && active) x[u] = __ldg(tab + (int64_t)r[u] * nvec + vi);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float f[E];
                    unpack16<DT>(x[u], f);
                    if constexpr (KAHAN) {
                        if (r[u] >= 0) {
#pragma unroll
                            for (int e = 0; e < E; ++e) {
                                const float y = fmaf(w[u], f[e], -comp[e]);
                                const float t = acc[e] + y;
                                comp[e] = (t - acc[e]) - y;
                                acc[e] = t;
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < E; e += 2)  // packed: each half rounds like fmaf
                            ffma2(acc[e], acc[e + 1], w[u], f[e], f[e + 1]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            cr[j] = nr[j];
            cw[j] = nw[j];
        }
    }
}

// Write this lane's vector vi of a pooled row, dividing by L for mean pooling.
template <int DT>
__device__ __forceinline__ void write_vec(float* __restrict__ orow, const float (&acc)[VecTraits<DT>::E],
                                          int nvec, int vi, int64_t L, bool mean, bool vec_out) {
    constexpr int E = VecTraits<DT>::E;
    if (vi >= nvec) return;
    const float Lf = (float)L;
    const bool div = mean && L > 0;
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = div ? __fdiv_rn(acc[e], Lf) : acc[e];
    float* dst = orow + (int64_t)vi * E;
    if (vec_out) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q)
            reinterpret_cast<float4*>(dst)[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = o[e];
    }
}

template <int G, int DT, typename IDX>
__device__ __forceinline__ void pool_bag_vec(const TableDesc& td, const FwdArgs& a, int64_t start, int64_t end,
                                             float* orow, int vi, int sub, unsigned mask, bool& oob) {
    constexpr int E = VecTraits<DT>::E;
    float acc[E], comp[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = comp[e] = 0.f;
    const int nvec = td.row_bytes >> 4;
    gather_accumulate<G, DT, IDX, false>(reinterpret_cast<const uint4*>(td.data), nvec, vi, td.rows,
                                         reinterpret_cast<const IDX*>(a.indices), a.weights, start, end, sub,
                                         mask, acc, comp, oob);
    write_vec<DT>(orow, acc, nvec, vi, end - start, a.mean != 0, a.vec_out != 0);
}

template <int DT, typename IDX>
__device__ __forceinline__ void pool_bag_vec_dispatch(const TableDesc& td, const FwdArgs& a, int64_t start,
                                                      int64_t end, float* orow, int vi, int sub, unsigned mask,
                                                      bool& oob) {
    switch (td.lanes) {
        case 1: pool_bag_vec<1, DT, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
        case 2: pool_bag_vec<2, DT, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
        case 4: pool_bag_vec<4, DT, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
        case 8: pool_bag_vec<8, DT, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
        case 16: pool_bag_vec<16, DT, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
        default: pool_bag_vec<32, DT, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
    }
}

// Element-wise path (rows that are not whole 16-byte vectors): one warp per
// bag, lane owns columns lane + 32q of each 128-column block.
template <int DT, typename IDX, bool KAHAN>
__device__ void sum_bag_scalar(const TableDesc& td, const FwdArgs& a, int64_t start, int64_t end, int cb,
                               int lane, float (&acc)[4], bool& oob) {
    const IDX* indices = reinterpret_cast<const IDX*>(a.indices);
    const int D = td.dim;
    float comp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = 0.f;
    for (int64_t c0 = start; c0 < end; c0 += 32) {
        const int64_t p = c0 + lane;
        int r = -1;
        float w = 1.f;
        if (p < end) {
            const int64_t x = ld_index(indices, p);
            if (x >= 0 && x < td.rows)
                r = (int)x;
            else
                oob = true;
            if (a.weights) w = __ldg(a.weights + p);
        }
        const int n = (int)tmin<int64_t>(32, end - c0);
        for (int k = 0; k < n; ++k) {
            const int rk = __shfl_sync(0xffffffffu, r, k);
            const float wk = __shfl_sync(0xffffffffu, w, k);
            if (rk < 0) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int col = cb + lane + 32 * q;
                if (col < D) {
                    const float f = load_elem<DT>(td.data, (int64_t)rk * D + col);
                    if constexpr (KAHAN) {
                        const float y = fmaf(wk, f, -comp[q]);
                        const float t = acc[q] + y;
                        comp[q] = (t - acc[q]) - y;
                        acc[q] = t;
                    } else {
                        acc[q] = fmaf(wk, f, acc[q]);
                    }
                }
            }
        }
    }
}

template <int DT, typename IDX>
__device__ void pool_bag_scalar(const TableDesc& td, const FwdArgs& a, int64_t start, int64_t end,
                                float* orow, int lane, bool& oob) {
    const int D = td.dim;
    const int64_t L = end - start;
    for (int cb = 0; cb < D; cb += 128) {
        float acc[4];
        sum_bag_scalar<DT, IDX, false>(td, a, start, end, cb, lane, acc, oob);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int col = cb + lane + 32 * q;
            if (col < D) orow[col] = (a.mean && L > 0) ? __fdiv_rn(acc[q], (float)L) : acc[q];
        }
    }
}

// Reads and checks one bag's [start, end).  Malformed offsets raise
// ERR_OFFSETS and the bag is treated as empty.
template <typename IDX>
__device__ __forceinline__ void bag_range(const FwdArgs& a, int64_t bag, int64_t& start, int64_t& end,
                                          bool report) {
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    start = ld_index(off, bag);
    end = ld_index(off, bag + 1);
    const int64_t nb = (int64_t)a.T * a.B;
    bool bad = start < 0 || end < start || end > a.N;
    if (bag == 0 && start != 0) bad = true;
    if (bag == nb - 1 && end != a.N) bad = true;
    if (bad) {
        if (report) atomicOr(&a.blk->error, ERR_OFFSETS);
        start = end = 0;
    }
}

template <typename IDX>
__global__ void __launch_bounds__(256, 4) fwd_pool_kernel(FwdArgs a) {
    chain_wait();  // returns at once unless launched chained (after the bag order)
    const int gw = (int)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (gw >= a.total_warps) return;
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = a.T - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.tabs[mid].warp_begin <= gw)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int t = lo;
    const TableDesc td = a.tabs[t];
    const bool vec = td.path == PATH_VEC;
    const int G = vec ? td.lanes : 32;
    const int ncb = vec ? td.vecs : 1;  // column blocks of 32 vectors
    const int slot = lane / G, sub = lane % G;
    const int w = gw - td.warp_begin;
    const int cb = w % ncb;
    int b = (w / ncb) * (32 / G) + slot;
    if (b >= a.B) return;  // the whole slot leaves together
    // length-keyed order: slot b takes the table's b-th bag by length
    if (a.order && a.lflag[t]) {
        const uint32_t ob = __ldg(a.order + (int64_t)t * a.B + b);
        if (ob >= (uint32_t)a.B) return;  // (a permutation of the table's bags: never taken)
        b = (int)ob;
    }
    const unsigned mask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (slot * G));
    const int64_t bag = (int64_t)t * a.B + b;
    int64_t start, end;
    bag_range<IDX>(a, bag, start, end, sub == 0 && cb == 0);
    float* orow = a.out + (int64_t)b * a.total_d + td.doff;
    bool oob = false;
    if (end - start > kLongBag) {
        // queued once (by column block 0) for the CTA kernel; if the queue is
        // full, column block 0 pools every column block of the bag itself
        if (cb != 0) return;
        int queued = 0;
        if (sub == 0) {
            const uint32_t k = atomicAdd(&a.blk->long_count[a.parity], 1u);
            if (k < (uint32_t)kLongBagCap) {
                a.blk->long_bags[a.parity][k] = (uint64_t)bag;
                queued = 1;
            }
        }
        queued = __shfl_sync(mask, queued, 0, G);
        if (queued) return;
        if (vec) {
            for (int c = 0; c < ncb; ++c) {
                switch (td.dtype) {
                    case DT_F32: pool_bag_vec_dispatch<DT_F32, IDX>(td, a, start, end, orow, c * 32 + sub, sub, mask, oob); break;
                    case DT_F16: pool_bag_vec_dispatch<DT_F16, IDX>(td, a, start, end, orow, c * 32 + sub, sub, mask, oob); break;
                    default: pool_bag_vec_dispatch<DT_BF16, IDX>(td, a, start, end, orow, c * 32 + sub, sub, mask, oob); break;
                }
            }
            if (__any_sync(mask, oob) && sub == 0) atomicOr(&a.blk->error, ERR_OOB);
            return;
        }
    }
    if (vec) {
        const int vi = cb * 32 + sub;
        switch (td.dtype) {
            case DT_F32: pool_bag_vec_dispatch<DT_F32, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
            case DT_F16: pool_bag_vec_dispatch<DT_F16, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
            default: pool_bag_vec_dispatch<DT_BF16, IDX>(td, a, start, end, orow, vi, sub, mask, oob); break;
        }
    } else {
        switch (td.dtype) {
            case DT_F32: pool_bag_scalar<DT_F32, IDX>(td, a, start, end, orow, lane, oob); break;
            case DT_F16: pool_bag_scalar<DT_F16, IDX>(td, a, start, end, orow, lane, oob); break;
            default: pool_bag_scalar<DT_BF16, IDX>(td, a, start, end, orow, lane, oob); break;
        }
    }
    if (__any_sync(mask, oob) && sub == 0) atomicOr(&a.blk->error, ERR_OOB);
}

// ---------------------------------------------------------------- long bags

constexpr int kLongWarps = 8;
constexpr int kLongMaxFloats = 1024;  // floats of one row held per warp in shared memory

template <int DT, typename IDX>
__device__ void long_bag_vec(const TableDesc& td, const FwdArgs& a, int64_t start, int64_t end, float* orow,
                             float (*part)[kLongMaxFloats], bool& oob) {
    constexpr int E = VecTraits<DT>::E;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = td.row_bytes >> 4;
    const int64_t L = end - start;
    const int64_t s0 = start + L * warp / kLongWarps;
    const int64_t s1 = start + L * (warp + 1) / kLongWarps;
    for (int cb = 0; cb * 32 < nvec; ++cb) {
        const int vi = cb * 32 + lane;
        float acc[E], comp[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = comp[e] = 0.f;
        gather_accumulate<32, DT, IDX, true>(reinterpret_cast<const uint4*>(td.data), nvec, vi, td.rows,
                                             reinterpret_cast<const IDX*>(a.indices), a.weights, s0, s1, lane,
                                             0xffffffffu, acc, comp, oob);
        if (vi < nvec)
#pragma unroll
            for (int e = 0; e < E; ++e) part[warp][vi * E + e] = acc[e] - comp[e];
    }
    __syncthreads();
    const int D = td.dim;
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float s = 0.f, cmp = 0.f;
#pragma unroll
        for (int w = 0; w < kLongWarps; ++w) {  // fixed order
            const float y = part[w][c] - cmp;
            const float t = s + y;
            cmp = (t - s) - y;
            s = t;
        }
        s -= cmp;
        orow[c] = (a.mean && L > 0) ? __fdiv_rn(s, (float)L) : s;
    }
    __syncthreads();
}

template <int DT, typename IDX>
__device__ void long_bag_scalar(const TableDesc& td, const FwdArgs& a, int64_t start, int64_t end,
                                float* orow, float (*part)[kLongMaxFloats], bool& oob) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = td.dim;
    const int64_t L = end - start;
    const int64_t s0 = start + L * warp / kLongWarps;
    const int64_t s1 = start + L * (warp + 1) / kLongWarps;
    for (int cb = 0; cb < D; cb += 128) {
        float acc[4];
        sum_bag_scalar<DT, IDX, true>(td, a, s0, s1, cb, lane, acc, oob);
#pragma unroll
        for (int q = 0; q < 4; ++q) part[warp][lane + 32 * q] = acc[q];
        __syncthreads();
        for (int c = threadIdx.x; c < 128 && cb + c < D; c += blockDim.x) {
            float s = 0.f, cmp = 0.f;
#pragma unroll
            for (int w = 0; w < kLongWarps; ++w) {
                const float y = part[w][c] - cmp;
                const float t = s + y;
                cmp = (t - s) - y;
                s = t;
            }
            s -= cmp;
            orow[cb + c] = (a.mean && L > 0) ? __fdiv_rn(s, (float)L) : s;
        }
        __syncthreads();
    }
}

template <typename IDX>
__global__ void __launch_bounds__(256) fwd_long_kernel(FwdArgs a) {
    chain_wait();  // returns at once unless launched chained
    __shared__ float part[kLongWarps][kLongMaxFloats];
    const uint32_t cnt = tmin(*(volatile uint32_t*)&a.blk->long_count[a.parity], (uint32_t)kLongBagCap);
    bool oob = false;
    for (uint32_t i = blockIdx.x; i < cnt; i += gridDim.x) {
        const int64_t bag = (int64_t)a.blk->long_bags[a.parity][i];
        const int t = (int)(bag / a.B);
        const int b = (int)(bag - (int64_t)t * a.B);
        const TableDesc td = a.tabs[t];
        int64_t start, end;
        bag_range<IDX>(a, bag, start, end, false);
        float* orow = a.out + (int64_t)b * a.total_d + td.doff;
        if (td.path == PATH_VEC) {
            switch (td.dtype) {
                case DT_F32: long_bag_vec<DT_F32, IDX>(td, a, start, end, orow, part, oob); break;
                case DT_F16: long_bag_vec<DT_F16, IDX>(td, a, start, end, orow, part, oob); break;
                default: long_bag_vec<DT_BF16, IDX>(td, a, start, end, orow, part, oob); break;
            }
        } else {
            switch (td.dtype) {
                case DT_F32: long_bag_scalar<DT_F32, IDX>(td, a, start, end, orow, part, oob); break;
                case DT_F16: long_bag_scalar<DT_F16, IDX>(td, a, start, end, orow, part, oob); break;
                default: long_bag_scalar<DT_BF16, IDX>(td, a, start, end, orow, part, oob); break;
            }
        }
    }
    if (oob) atomicOr(&a.blk->error, ERR_OOB);
    // The next call uses the other counter; it was last read by the previous
    // call's long kernel, which has finished (same stream).
    if (blockIdx.x == 0 && threadIdx.x == 0) a.blk->long_count[a.parity ^ 1] = 0;
}

// ------------------------------------------------------ length-keyed order
//
// A warp pools 32/G bags side by side and a CTA holds its SM slot until its
// longest bag is done, so bags of very different lengths in one CTA leave
// most of its lanes idle.  When a table's bags differ in length, its bags
// are taken in order of length instead (a counting sort per table: lengths
// bucketed, kLenBuckets buckets), so each CTA's bags are about equally long.
// Each bag's result does not depend on which slot pools it.

// Both kernels run one CTA per chunk of kOrderChunk bags of one table
// (grid T x chunks); lcount and ldone are zero between calls (the last CTA
// of each table clears them).
constexpr int kOrderChunk = 4096;

// Length bucket of bag b of table t.
template <typename IDX>
__device__ __forceinline__ uint32_t bag_len_bucket(const FwdArgs& a, int t, int b) {
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const int64_t g = (int64_t)t * a.B + b;
    const int64_t len = ld_index(off, g + 1) - ld_index(off, g);
    return len < 0 ? 0u : (len >= kLenBuckets - 1 ? (uint32_t)(kLenBuckets - 1) : (uint32_t)len);
}

// Counts the chunk's bags per length bucket (shared memory, one atomic per
// group of equal buckets in a warp) into lcount[t]; the table's last CTA
// turns the counts into the buckets' first ranks and sets lflag[t] when the
// table's bags have more than one length.
template <typename IDX>
__global__ void __launch_bounds__(256) bag_len_count_kernel(FwdArgs a, int chunks) {
    __shared__ uint32_t s_cnt[kLenBuckets];
    __shared__ uint32_t s_last;
    const int t = (int)(blockIdx.x / (unsigned)chunks), j = (int)(blockIdx.x % (unsigned)chunks);
    const int lane = threadIdx.x & 31;
    if (a.tabs[t].path == PATH_HIST) {
        if (j == 0 && threadIdx.x == 0) a.lflag[t] = 0u;
        return;
    }
    for (int k = threadIdx.x; k < kLenBuckets; k += blockDim.x) s_cnt[k] = 0u;
    __syncthreads();
    const int b0 = j * kOrderChunk, b1 = tmin<int>(a.B, b0 + kOrderChunk);
    for (int base = b0; base < b1; base += blockDim.x) {  // whole warps together
        const int b = base + threadIdx.x;
        const uint32_t l = b < b1 ? bag_len_bucket<IDX>(a, t, b) : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, l);
        if (l != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&s_cnt[l], (uint32_t)__popc(peers));
    }
    __syncthreads();
    uint32_t* c = a.lcount + (int64_t)t * kLenBuckets;
    for (int k = threadIdx.x; k < kLenBuckets; k += blockDim.x)
        if (s_cnt[k]) atomicAdd(c + k, s_cnt[k]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.ldone + t, 1u) == (uint32_t)chunks - 1u;
    __syncthreads();
    if (!s_last) return;
    // last CTA of the table: exclusive scan of the counts (warp 0)
    __threadfence();
    if (threadIdx.x < 32) {
        constexpr int P = kLenBuckets / 32;
        uint32_t v[P], sum = 0, nz = 0;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            v[i] = __ldcg(c + lane * P + i);
            sum += v[i];
            nz += v[i] != 0u;
        }
        uint32_t x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) nz += __shfl_xor_sync(0xffffffffu, nz, o);
        uint32_t run = x - sum;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            c[lane * P + i] = run;
            run += v[i];
        }
        if (lane == 0) {
            a.lflag[t] = nz > 1u ? 1u : 0u;
            a.ldone[t] = 0u;
        }
    }
}

// Every bag of a table with lflag set gets its rank: its bucket's next free
// one (a warp's bags of one bucket take consecutive ranks in lane order).
// The table's last CTA clears lcount[t] (and the first CTA does when the
// table keeps index order).
template <typename IDX>
__global__ void __launch_bounds__(256) bag_len_order_kernel(FwdArgs a, int chunks) {
    chain_wait();
    __shared__ uint32_t s_last;
    const int t = (int)(blockIdx.x / (unsigned)chunks), j = (int)(blockIdx.x % (unsigned)chunks);
    const int lane = threadIdx.x & 31;
    if (a.tabs[t].path == PATH_HIST) return;
    uint32_t* c = a.lcount + (int64_t)t * kLenBuckets;
    if (!a.lflag[t]) {
        if (j == 0)
            for (int k = threadIdx.x; k < kLenBuckets; k += blockDim.x) c[k] = 0u;
        return;
    }
    const int b0 = j * kOrderChunk, b1 = tmin<int>(a.B, b0 + kOrderChunk);
    for (int base = b0; base < b1; base += blockDim.x) {  // whole warps together
        const int b = base + threadIdx.x;
        const uint32_t l = b < b1 ? bag_len_bucket<IDX>(a, t, b) : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, l);
        const int leader = __ffs(peers) - 1;
        uint32_t r0 = 0;
        if (l != 0xffffffffu && lane == leader) r0 = atomicAdd(c + l, (uint32_t)__popc(peers));
        r0 = __shfl_sync(0xffffffffu, r0, leader);
        if (l != 0xffffffffu) {
            const uint32_t r = r0 + (uint32_t)__popc(peers & ((1u << lane) - 1u));
            if (r < (uint32_t)a.B) a.order[(int64_t)t * a.B + r] = (uint32_t)b;
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.ldone + t, 1u) == (uint32_t)chunks - 1u;
    __syncthreads();
    if (!s_last) return;
    for (int k = threadIdx.x; k < kLenBuckets; k += blockDim.x) c[k] = 0u;
    if (threadIdx.x == 0) a.ldone[t] = 0u;
}

// Warp map for batch size B: warp_begin[t] = sum over earlier non-histogram
// tables of ceil(B / (32 / G_u)) * blocks_u.  One small CTA, launched when B
// changes.
__global__ void fwd_schedule_kernel(TableDesc* tabs, int T, int B) {
    if (threadIdx.x != 0) return;
    int acc = 0;
    for (int t = 0; t < T; ++t) {
        tabs[t].warp_begin = acc;
        if (tabs[t].path == PATH_HIST) continue;
        const bool vec = tabs[t].path == PATH_VEC;
        const int per = vec ? 32 / tabs[t].lanes : 1;
        const int blocks = vec ? tabs[t].vecs : 1;
        acc += (B + per - 1) / per * blocks;
    }
}

cudaError_t launch_forward_schedule(TableDesc* tabs, int T, int B, cudaStream_t s) {
    fwd_schedule_kernel<<<1, 32, 0, s>>>(tabs, T, B);
    return cudaGetLastError();
}

// The length-keyed order (count with scan, then rank): two kernels on s; a
// kernel that reads the order should follow them chained.
cudaError_t launch_bag_order(const FwdArgs& a, cudaStream_t s) {
    const int chunks = (a.B + kOrderChunk - 1) / kOrderChunk;
    const unsigned ogrid = (unsigned)((int64_t)a.T * chunks);
    if (a.idx64)
        bag_len_count_kernel<int64_t><<<ogrid, 256, 0, s>>>(a, chunks);
    else
        bag_len_count_kernel<int32_t><<<ogrid, 256, 0, s>>>(a, chunks);
    return a.idx64 ? launch_chained(bag_len_order_kernel<int64_t>, dim3(ogrid), dim3(256), s, a, chunks)
                   : launch_chained(bag_len_order_kernel<int32_t>, dim3(ogrid), dim3(256), s, a, chunks);
}

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s) {
    if (a.total_warps > 0) {
        const bool ordered = a.order != nullptr;
        if (ordered) {
            const cudaError_t e = launch_bag_order(a, s);
            if (e != cudaSuccess) return e;
        }
        const int64_t threads = (int64_t)a.total_warps * 32;
        const unsigned grid = (unsigned)((threads + 255) / 256);
        cudaError_t e;
        if (ordered) {
            e = a.idx64 ? launch_chained(fwd_pool_kernel<int64_t>, dim3(grid), dim3(256), s, a)
                        : launch_chained(fwd_pool_kernel<int32_t>, dim3(grid), dim3(256), s, a);
        } else {
            if (a.idx64)
                fwd_pool_kernel<int64_t><<<grid, 256, 0, s>>>(a);
            else
                fwd_pool_kernel<int32_t><<<grid, 256, 0, s>>>(a);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
    }
    const unsigned lgrid = (unsigned)(a.num_sms > 0 ? a.num_sms : 1);
    if (a.total_warps > 0)  // chained after the pooling kernel
        return a.idx64 ? launch_chained(fwd_long_kernel<int64_t>, dim3(lgrid), dim3(256), s, a)
                       : launch_chained(fwd_long_kernel<int32_t>, dim3(lgrid), dim3(256), s, a);
    if (a.idx64)
        fwd_long_kernel<int64_t><<<lgrid, 256, 0, s>>>(a);
    else
        fwd_long_kernel<int32_t><<<lgrid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tbe
