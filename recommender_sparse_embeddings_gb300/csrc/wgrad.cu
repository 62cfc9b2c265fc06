// Gradient of the loss with respect to the per-sample weights (kimbodo "What
// Happened": the generic path takes per-sample weights; when they are trained
// they need their own gradient).  The forward pass computes
//   out[b, Doff_t + j] = (1/L if mean) * sum_{i in bag(t,b)} w_i W_t[idx_i, j],
// so for every lookup i of bag (t, b)
//   dL/dw_i = (1/L if mean) * sum_j G[b, Doff_t + j] * W_t[idx_i, j],
// a dot product of the looked-up row, as stored before this step's update,
// with the bag's slice of the upstream gradient G.  A lookup whose index is
// out of range is skipped by the forward pass, so its gradient is 0.
//
// Schedule: one warp per bag.  Rows that are whole 16-byte vectors use the
// forward pass's slot layout: a slot of G lanes covers 32 vectors of a row
// (one per lane), a warp holds 32/G slots and each slot takes every
// (32/G)-th lookup of the bag, four at a time (four CTAs of 256 per SM, 64
// registers: the gathers are latency bound).  Each lane keeps the bag's
// gradient for its vector in registers, multiplies it with the row's vector
// and the slot adds its lanes' partial dots in a fixed butterfly order.
// Other rows: the whole warp takes one lookup at a time, lane c owns columns
// c + 32q.  Reads: the looked-up rows (the same bytes as the forward pass),
// G once per bag, indices and offsets; writes: 4 bytes per lookup.
#include "tbe_internal.cuh"

namespace tbe {

namespace {

template <int DT>
struct WVec {
    static constexpr int E = (DT == DT_F32) ? 4 : 8;  // elements per 16-byte vector
};

// Reads and checks one bag's [start, end), the forward pass's rule: a
// malformed bag reports ERR_OFFSETS and counts as empty.
template <typename IDX>
__device__ __forceinline__ void wg_bag_range(const WgradArgs& a, int64_t bag, int64_t& start, int64_t& end,
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

// E gradient values of vector vi of the bag's slice (zeros past the row).
template <int E>
__device__ __forceinline__ void load_gvec(const float* __restrict__ grow, int vi, int nvec, bool vec,
                                          float (&g)[E]) {
#pragma unroll
    for (int e = 0; e < E; ++e) g[e] = 0.f;
    if (vi >= nvec) return;
    const float* p = grow + (int64_t)vi * E;
    if (vec) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p) + q);
            g[4 * q] = v.x;
            g[4 * q + 1] = v.y;
            g[4 * q + 2] = v.z;
            g[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) g[e] = __ldg(p + e);
    }
}

template <int G, int DT, typename IDX>
__device__ void wgrad_bag_vec(const TableDesc& td, const WgradArgs& a, int b, int64_t start, int64_t end, int lane,
                              bool& oob) {
    constexpr int E = WVec<DT>::E;
    constexpr int S = 32 / G;  // slots per warp
    constexpr int U = 4;       // lookups in flight per slot
    const int slot = lane / G, sub = lane % G;
    const unsigned mask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (slot * G));
    const int nvec = td.row_bytes >> 4, ncb = td.vecs;
    const float* grow = a.grad + (int64_t)b * a.total_d + td.doff;
    const bool gv = a.grad_vec && td.doff % 4 == 0;
    const uint4* tab = reinterpret_cast<const uint4*>(td.data);
    const IDX* indices = reinterpret_cast<const IDX*>(a.indices);
    const int64_t L = end - start;
    float g0[E];  // column block 0 of the bag's gradient, held for the whole bag
    load_gvec<E>(grow, sub, nvec, gv, g0);
    for (int64_t p0 = start + slot; p0 < end; p0 += (int64_t)S * U) {
        int r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t p = p0 + (int64_t)u * S;
            r[u] = -1;
            if (p < end) {
                const int64_t x = ld_index(indices, p);  // the slot's lanes read one address
                if (x >= 0 && x < td.rows)
                    r[u] = (int)x;
                else
                    oob = true;
            }
        }
        float dot[U];
#pragma unroll
        for (int u = 0; u < U; ++u) dot[u] = 0.f;
        for (int cb = 0; cb < ncb; ++cb) {
            const int vi = cb * 32 + sub;
            float g[E];
            if (cb == 0) {
#pragma unroll
                for (int e = 0; e < E; ++e) g[e] = g0[e];
            } else {
                load_gvec<E>(grow, vi, nvec, gv, g);
            }
            uint4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                x[u] = make_uint4(0u, 0u, 0u, 0u);
                if (r[u] >= 0 && vi < nvec) x[u] = __ldg(tab + (int64_t)r[u] * nvec + vi);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float f[E];
                unpack16<DT>(x[u], f);
#pragma unroll
                for (int e = 0; e < E; ++e) dot[u] = fmaf(g[e], f[e], dot[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) dot[u] += __shfl_xor_sync(mask, dot[u], o, G);
        }
        if (sub == 0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t p = p0 + (int64_t)u * S;
                if (p < end) {
                    float v = r[u] >= 0 ? dot[u] : 0.f;
                    if (a.mean && L > 0) v = __fdiv_rn(v, (float)L);
                    a.out[p] = v;
                }
            }
        }
    }
}

template <int DT, typename IDX>
__device__ void wgrad_bag_scalar(const TableDesc& td, const WgradArgs& a, int b, int64_t start, int64_t end,
                                 int lane, bool& oob) {
    const IDX* indices = reinterpret_cast<const IDX*>(a.indices);
    const int D = td.dim;
    const float* grow = a.grad + (int64_t)b * a.total_d + td.doff;
    const int64_t L = end - start;
    for (int64_t p = start; p < end; ++p) {
        const int64_t x = ld_index(indices, p);
        const bool ok = x >= 0 && x < td.rows;
        if (!ok) oob = true;
        float dot = 0.f;
        if (ok) {
            for (int c = lane; c < D; c += 32)
                dot = fmaf(__ldg(grow + c), load_elem<DT>(td.data, x * D + c), dot);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) {
            float v = ok ? dot : 0.f;
            if (a.mean && L > 0) v = __fdiv_rn(v, (float)L);
            a.out[p] = v;
        }
    }
}

template <int DT, typename IDX>
__device__ __forceinline__ void wgrad_bag(const TableDesc& td, const WgradArgs& a, int b, int64_t start,
                                          int64_t end, int lane, bool& oob) {
    const bool vec = td.row_bytes % 16 == 0 && ((uintptr_t)td.data % 16) == 0 && (td.row_bytes >> 4) <= 128;
    if (!vec) {
        wgrad_bag_scalar<DT, IDX>(td, a, b, start, end, lane, oob);
        return;
    }
    switch (td.lanes) {
        case 1: wgrad_bag_vec<1, DT, IDX>(td, a, b, start, end, lane, oob); break;
        case 2: wgrad_bag_vec<2, DT, IDX>(td, a, b, start, end, lane, oob); break;
        case 4: wgrad_bag_vec<4, DT, IDX>(td, a, b, start, end, lane, oob); break;
        case 8: wgrad_bag_vec<8, DT, IDX>(td, a, b, start, end, lane, oob); break;
        case 16: wgrad_bag_vec<16, DT, IDX>(td, a, b, start, end, lane, oob); break;
        default: wgrad_bag_vec<32, DT, IDX>(td, a, b, start, end, lane, oob); break;
    }
}

template <typename IDX>
__global__ void __launch_bounds__(256, 4) wgrad_kernel(WgradArgs a) {
    chain_wait();  // returns at once unless launched chained (after the bag order)
    int64_t bag = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // one warp per bag
    if (bag >= (int64_t)a.T * a.B) return;
    const int lane = threadIdx.x & 31;
    const int t = (int)(bag / a.B);
    int b = (int)(bag - (int64_t)t * a.B);
    // length-keyed order: warp b takes the table's b-th bag by length
    if (a.order && a.lflag[t]) {
        const uint32_t ob = __ldg(a.order + bag);
        if (ob >= (uint32_t)a.B) return;  // (a permutation of the table's bags: never taken)
        b = (int)ob;
        bag = (int64_t)t * a.B + b;
    }
    const TableDesc td = a.tabs[t];
    int64_t start, end;
    wg_bag_range<IDX>(a, bag, start, end, lane == 0);
    bool oob = false;
    switch (td.dtype) {
        case DT_F32: wgrad_bag<DT_F32, IDX>(td, a, b, start, end, lane, oob); break;
        case DT_F16: wgrad_bag<DT_F16, IDX>(td, a, b, start, end, lane, oob); break;
        default: wgrad_bag<DT_BF16, IDX>(td, a, b, start, end, lane, oob); break;
    }
    if (__any_sync(0xffffffffu, oob) && lane == 0) atomicOr(&a.blk->error, ERR_OOB);
}

}  // namespace

cudaError_t launch_wgrad(const WgradArgs& a, cudaStream_t s) {
    const int64_t warps = (int64_t)a.T * a.B;
    if (warps == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    if (a.order)
        return a.idx64 ? launch_chained(wgrad_kernel<int64_t>, dim3(blocks), dim3(256), s, a)
                       : launch_chained(wgrad_kernel<int32_t>, dim3(blocks), dim3(256), s, a);
    if (a.idx64)
        wgrad_kernel<int64_t><<<blocks, 256, 0, s>>>(a);
    else
        wgrad_kernel<int32_t><<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tbe
