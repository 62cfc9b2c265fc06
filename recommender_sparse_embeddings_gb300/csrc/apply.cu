// Backward apply: per distinct (table,row) key, g = sum over its run of
// s_i * grad[bag_i, Doff_t : Doff_t + D_t] in fp32, then one optimizer update
// of that row (kimbodo "What Happened": one optimizer update per row, a
// streaming path for short runs, gradient accumulation for runs of at least
// 256 lookups).
//
//  short_runs_kernel: one warp per distinct key (persistent grid-stride).  A
//    run of fewer than kLongRun lookups is summed in order by that warp and
//    the row is updated in place.  A longer run is only registered: it gets
//    ceil(len/256) consecutive chunk slots.
//  long_chunks_kernel: one warp per 256-lookup chunk writes its partial sum;
//    the warp that completes the last chunk of a run (counted with an atomic
//    after a fence) adds the run's partials in chunk order and updates the
//    row.  Results do not depend on scheduling.
//
// Sums use compensated (Kahan) fp32 addition, so a run of 10^5 lookups keeps
// close to fp32 rounding of the exact sum.  Each lane owns VW consecutive
// columns of every 32*VW-column block, so the gradient rows are read with
// 4- to 16-byte loads across the warp.
#include "tbe_internal.cuh"

namespace tbe {

struct Kahan {
    float s, c;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ void add_scaled(float w, float x) {
        const float y = fmaf(w, x, -c);
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ float value() const { return s - c; }
};

__device__ __forceinline__ int table_of(const TableDesc* tabs, int T, uint32_t key) {
    int lo = 0, hi = T - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((uint64_t)tabs[mid].rowbase <= key)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Loads VW consecutive floats (VW*4 bytes, aligned) into f.
template <int VW>
__device__ __forceinline__ void ld_f32v(const float* p, float (&f)[VW]) {
    if constexpr (VW == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else if constexpr (VW == 2) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(p));
        f[0] = v.x; f[1] = v.y;
    } else {
        f[0] = __ldg(p);
    }
}

// Row slice of VW elements of dtype DT <-> floats (aligned vector access).
template <int DT, int VW>
__device__ __forceinline__ void ld_row(const void* base, int64_t k, float (&f)[VW]) {
    if constexpr (DT == DT_F32) {
        const float* p = reinterpret_cast<const float*>(base) + k;
        if constexpr (VW == 4) {
            const float4 v = *reinterpret_cast<const float4*>(p);
            f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
        } else if constexpr (VW == 2) {
            const float2 v = *reinterpret_cast<const float2*>(p);
            f[0] = v.x; f[1] = v.y;
        } else {
            f[0] = *p;
        }
    } else {
        const unsigned short* p = reinterpret_cast<const unsigned short*>(base) + k;
        uint32_t w[(VW + 1) / 2];
        if constexpr (VW == 4) {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            w[0] = v.x; w[1] = v.y;
        } else if constexpr (VW == 2) {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        } else {
            w[0] = *p;
        }
#pragma unroll
        for (int i = 0; i < VW; ++i) {
            const uint32_t h = (w[i / 2] >> (16 * (i & 1))) & 0xffffu;
            f[i] = DT == DT_F16 ? h_bits_to_float(h) : bf16_bits_to_float(h);
        }
    }
}

template <int DT, int VW>
__device__ __forceinline__ void st_row(void* base, int64_t k, const float (&f)[VW]) {
    if constexpr (DT == DT_F32) {
        float* p = reinterpret_cast<float*>(base) + k;
        if constexpr (VW == 4)
            *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
        else if constexpr (VW == 2)
            *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
        else
            *p = f[0];
    } else {
        uint32_t h[VW];
#pragma unroll
        for (int i = 0; i < VW; ++i) {
            if constexpr (DT == DT_F16)
                h[i] = __half_as_ushort(__float2half_rn(f[i]));
            else
                h[i] = __bfloat16_as_ushort(__float2bfloat16_rn(f[i]));
        }
        unsigned short* p = reinterpret_cast<unsigned short*>(base) + k;
        if constexpr (VW == 4)
            *reinterpret_cast<uint2*>(p) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        else if constexpr (VW == 2)
            *reinterpret_cast<uint32_t*>(p) = h[0] | (h[1] << 16);
        else
            *p = (unsigned short)h[0];
    }
}

// Column layout of a row of D floats for one warp: NB blocks of 32*VW
// columns; lane owns columns blk*32*VW + lane*VW + [0, VW).
template <int VW, int NB>
struct Cols {
    static constexpr int N = VW * NB;
    __device__ __forceinline__ static int col(int lane, int blk) { return blk * 32 * VW + lane * VW; }
};

// Sum of s_i * grad rows over sorted slots [s0, s1) into acc (per lane).
template <int VW, int NB>
__device__ __forceinline__ void reduce_run(const ApplyArgs& a, const Workspace& ws, const uint32_t* __restrict__ pos_sorted,
                                           int t, int doff, uint32_t s0, uint32_t s1, int lane,
                                           Kahan (&acc)[NB][VW]) {
    constexpr int U = 4;
    const int64_t tB = (int64_t)t * a.B;
    const int64_t nbags = (int64_t)a.T * a.B;
    for (uint32_t c0 = s0; c0 < s1; c0 += 32) {
        const uint32_t i = c0 + lane;
        int64_t b = -1;
        float s = 1.f;
        if (i < s1) {
            const uint32_t pos = __ldg(pos_sorted + i);
            if (pos < (uint32_t)a.N) {
                const uint32_t bag = __ldg(ws.bag + pos);
                if ((int64_t)bag < nbags && (int64_t)bag >= tB && (int64_t)bag < tB + a.B) b = bag - tB;
                if (a.has_scale) s = __ldg(ws.scale + pos);
            }
        }
        const int n = (int)tmin<uint32_t>(32u, s1 - c0);
        for (int k0 = 0; k0 < n; k0 += U) {
            int64_t bb[U];
            float ss[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                bb[u] = __shfl_sync(0xffffffffu, b, (k0 + u) & 31);
                ss[u] = __shfl_sync(0xffffffffu, s, (k0 + u) & 31);
                if (k0 + u >= n) bb[u] = -1;
            }
            float g[U][NB][VW];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int q = 0; q < NB; ++q) {
                    if (bb[u] >= 0) {
                        ld_f32v<VW>(a.grad + bb[u] * a.total_d + doff + Cols<VW, NB>::col(lane, q), g[u][q]);
                    } else {
#pragma unroll
                        for (int v = 0; v < VW; ++v) g[u][q][v] = 0.f;
                    }
                }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (bb[u] >= 0)
#pragma unroll
                    for (int q = 0; q < NB; ++q)
#pragma unroll
                        for (int v = 0; v < VW; ++v) acc[q][v].add_scaled(ss[u], g[u][q][v]);
        }
    }
}

// One optimizer step on row r of table t with gradient g (this lane's columns).
template <int DT, int VW, int NB>
__device__ __forceinline__ void update_row(const ApplyArgs& a, const TableDesc& td, uint32_t key,
                                           int64_t r, const float (&g)[NB][VW], int lane) {
    float step[NB][VW];
    if (a.opt == 2) {
        float sq = 0.f;
#pragma unroll
        for (int q = 0; q < NB; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v) sq = fmaf(g[q][v], g[q][v], sq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        const float m = a.state[key] + __fdiv_rn(sq, (float)td.dim);
        __syncwarp();
        if (lane == 0) a.state[key] = m;
        const float denom = sqrtf(m) + a.eps;
#pragma unroll
        for (int q = 0; q < NB; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v) step[q][v] = a.lr * __fdiv_rn(g[q][v], denom);
    } else {
#pragma unroll
        for (int q = 0; q < NB; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v) step[q][v] = a.lr * g[q][v];
    }
    const int64_t rowoff = r * td.dim;
#pragma unroll
    for (int q = 0; q < NB; ++q) {
        const int c = Cols<VW, NB>::col(lane, q);
        float w[VW];
        ld_row<DT, VW>(td.data, rowoff + c, w);
#pragma unroll
        for (int v = 0; v < VW; ++v) w[v] = w[v] - step[q][v];
        st_row<DT, VW>(td.data, rowoff + c, w);
    }
}

// Element-wise variant for dims that are not 32*VW*NB: lane owns columns
// lane + 32*j of each 256-column block.
template <int DT>
__device__ void reduce_update_generic(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos_sorted,
                                      const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                                      int lane, const float* partial_src, int nchunks) {
    const int D = td.dim;
    const int64_t r = (int64_t)key - td.rowbase;
    const int64_t tB = (int64_t)t * a.B;
    // Adagrad needs the whole row's sum of squares before any column moves:
    // first pass accumulates it, second pass recomputes g and updates.
    float sq = 0.f;
    for (int pass = 0; pass < (a.opt == 2 ? 2 : 1); ++pass) {
        float m = 0.f, denom = 1.f;
        if (a.opt == 2 && pass == 1) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
            m = a.state[key] + __fdiv_rn(sq, (float)D);
            denom = sqrtf(m) + a.eps;
        }
        for (int cb = 0; cb < D; cb += 256) {
            Kahan acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = Kahan{0.f, 0.f};
            if (partial_src) {
                for (int ch = 0; ch < nchunks; ++ch)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int c = cb + lane + 32 * j;
                        if (c < D) acc[j].add(__ldcg(partial_src + (int64_t)ch * a.max_dim + c));
                    }
            } else {
                for (uint32_t i = s0; i < s1; ++i) {
                    const uint32_t pos = __ldg(pos_sorted + i);
                    if (pos >= (uint32_t)a.N) continue;
                    const int64_t bag = __ldg(ws.bag + pos);
                    if (bag < tB || bag >= tB + a.B) continue;
                    const float s = a.has_scale ? __ldg(ws.scale + pos) : 1.f;
                    const float* grow = a.grad + (bag - tB) * a.total_d + td.doff;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int c = cb + lane + 32 * j;
                        if (c < D) acc[j].add_scaled(s, __ldg(grow + c));
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = cb + lane + 32 * j;
                if (c >= D) continue;
                const float g = acc[j].value();
                if (a.opt == 2 && pass == 0) {
                    sq = fmaf(g, g, sq);
                    continue;
                }
                const float step = a.opt == 2 ? a.lr * __fdiv_rn(g, denom) : a.lr * g;
                const float w = load_elem<DT>(td.data, r * D + c);
                store_elem<DT>(td.data, r * D + c, w - step);
            }
        }
        if (a.opt == 2 && pass == 1) {
            __syncwarp();
            if (lane == 0) a.state[key] = m;
        }
    }
}

template <int DT, int VW, int NB>
__device__ __forceinline__ void short_run(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos_sorted,
                                          const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                                          int lane) {
    Kahan acc[NB][VW];
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[q][v] = Kahan{0.f, 0.f};
    reduce_run<VW, NB>(a, ws, pos_sorted, t, td.doff, s0, s1, lane, acc);
    float g[NB][VW];
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) g[q][v] = acc[q][v].value();
    update_row<DT, VW, NB>(a, td, key, (int64_t)key - td.rowbase, g, lane);
}

// Dispatch on the row shape: dim = 32, 64, 128, 256 use vector lanes when the
// table rows and the gradient columns are aligned for them; anything else
// runs element-wise.  Codes: 1 -> (VW 1, NB 1), 2 -> (2, 1), 3 -> (4, 1),
// 4 -> (4, 2), 0 -> element-wise.
__device__ __forceinline__ int shape_code(const TableDesc& td, int total_d, bool grad_vec) {
    const bool rows16 = grad_vec && ((uintptr_t)td.data & 15u) == 0;
    const bool a4 = rows16 && (td.doff % 4 == 0) && (total_d % 4 == 0);
    const bool a2 = rows16 && (td.doff % 2 == 0) && (total_d % 2 == 0);
    if (td.dim == 32) return 1;
    if (td.dim == 64 && a2) return 2;
    if (td.dim == 128 && a4) return 3;
    if (td.dim == 256 && a4) return 4;
    return 0;
}

template <int DT>
__device__ void short_run_dispatch(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos_sorted,
                                   const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                                   int lane) {
    switch (shape_code(td, a.total_d, a.grad_vec != 0)) {
        case 1: short_run<DT, 1, 1>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
        case 2: short_run<DT, 2, 1>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
        case 3: short_run<DT, 4, 1>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
        case 4: short_run<DT, 4, 2>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
        default: reduce_update_generic<DT>(a, ws, pos_sorted, td, t, key, s0, s1, lane, nullptr, 0); break;
    }
}

__global__ void __launch_bounds__(256) short_runs_kernel(ApplyArgs a, Workspace ws, const uint32_t* pos_sorted) {
    a.has_scale = ws.counters[CTR_HAS_SCALE] != 0;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t U = tmin<uint32_t>(*(volatile uint32_t*)&ws.counters[CTR_U], (uint32_t)a.N);
    for (int64_t u = gw; u < U; u += nw) {
        const uint32_t key = __ldg(ws.uniq + u);
        if (key >= a.total_rows) continue;  // lookups with an index out of range
        const uint32_t s0 = __ldg(ws.runstart + u), s1 = __ldg(ws.runstart + u + 1);
        if (s1 > (uint32_t)a.N || s0 >= s1) continue;
        const uint32_t len = s1 - s0;
        if (len >= (uint32_t)kLongRun) {
            uint32_t base = 0, li = 0;
            const uint32_t nc = (len + kLongRun - 1) / kLongRun;
            if (lane == 0) {
                base = atomicAdd(&ws.counters[CTR_NCHUNK], nc);
                li = atomicAdd(&ws.counters[CTR_NLONG], 1u);
                if (li < ws.max_long && base + nc <= ws.max_chunks) {
                    ws.long_runs[4 * li + 0] = (uint32_t)u;
                    ws.long_runs[4 * li + 1] = base;
                    ws.long_runs[4 * li + 2] = nc;
                    ws.long_runs[4 * li + 3] = 0;  // chunks finished
                }
            }
            base = __shfl_sync(0xffffffffu, base, 0);
            li = __shfl_sync(0xffffffffu, li, 0);
            if (li < ws.max_long && base + nc <= ws.max_chunks)
                for (uint32_t j = lane; j < nc; j += 32) ws.chunk_run[base + j] = li;
            continue;
        }
        const int t = table_of(a.tabs, a.T, key);
        const TableDesc td = a.tabs[t];
        switch (td.dtype) {
            case DT_F32: short_run_dispatch<DT_F32>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
            case DT_F16: short_run_dispatch<DT_F16>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
            default: short_run_dispatch<DT_BF16>(a, ws, pos_sorted, td, t, key, s0, s1, lane); break;
        }
    }
}

// ------------------------------------------------------------- long runs

template <int DT, int VW, int NB>
__device__ void long_chunk(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos_sorted,
                           const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                           float* part_row, uint32_t li, int lane) {
    Kahan acc[NB][VW];
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[q][v] = Kahan{0.f, 0.f};
    reduce_run<VW, NB>(a, ws, pos_sorted, t, td.doff, s0, s1, lane, acc);
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) part_row[Cols<VW, NB>::col(lane, q) + v] = acc[q][v].value();
}

template <int DT, int VW, int NB>
__device__ void long_combine(const ApplyArgs& a, const TableDesc& td, uint32_t key, const float* part0,
                             uint32_t nc, int lane) {
    Kahan acc[NB][VW];
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[q][v] = Kahan{0.f, 0.f};
    for (uint32_t j = 0; j < nc; ++j) {
        const float* p = part0 + (int64_t)j * a.max_dim;
#pragma unroll
        for (int q = 0; q < NB; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v) acc[q][v].add(__ldcg(p + Cols<VW, NB>::col(lane, q) + v));
    }
    float g[NB][VW];
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) g[q][v] = acc[q][v].value();
    update_row<DT, VW, NB>(a, td, key, (int64_t)key - td.rowbase, g, lane);
}

template <int DT>
__device__ void long_dispatch(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos_sorted,
                              const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                              uint32_t chunk, uint32_t li, uint32_t base, uint32_t nc, int lane) {
    float* part_row = ws.partial + (int64_t)chunk * a.max_dim;
    const int code = shape_code(td, a.total_d, a.grad_vec != 0);
    // 1) this chunk's partial sum
    if (code == 0) {
        // element-wise: columns lane + 32*j, blocks of 256
        const int D = td.dim;
        const int64_t tB = (int64_t)t * a.B;
        for (int cb = 0; cb < D; cb += 256) {
            Kahan acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = Kahan{0.f, 0.f};
            for (uint32_t i = s0; i < s1; ++i) {
                const uint32_t pos = __ldg(pos_sorted + i);
                if (pos >= (uint32_t)a.N) continue;
                const int64_t bag = __ldg(ws.bag + pos);
                if (bag < tB || bag >= tB + a.B) continue;
                const float s = a.has_scale ? __ldg(ws.scale + pos) : 1.f;
                const float* grow = a.grad + (bag - tB) * a.total_d + td.doff;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = cb + lane + 32 * j;
                    if (c < D) acc[j].add_scaled(s, __ldg(grow + c));
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = cb + lane + 32 * j;
                if (c < D) part_row[c] = acc[j].value();
            }
        }
    } else if (code == 1) {
        long_chunk<DT, 1, 1>(a, ws, pos_sorted, td, t, key, s0, s1, part_row, li, lane);
    } else if (code == 2) {
        long_chunk<DT, 2, 1>(a, ws, pos_sorted, td, t, key, s0, s1, part_row, li, lane);
    } else if (code == 3) {
        long_chunk<DT, 4, 1>(a, ws, pos_sorted, td, t, key, s0, s1, part_row, li, lane);
    } else {
        long_chunk<DT, 4, 2>(a, ws, pos_sorted, td, t, key, s0, s1, part_row, li, lane);
    }
    // 2) the warp that finishes a run's last chunk combines all of them
    __threadfence();
    __syncwarp();
    uint32_t done = 0;
    if (lane == 0) done = atomicAdd(&ws.long_runs[4 * li + 3], 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done != nc - 1) return;
    __threadfence();
    const float* part0 = ws.partial + (int64_t)base * a.max_dim;
    switch (code) {
        case 0: reduce_update_generic<DT>(a, ws, pos_sorted, td, t, key, 0, 0, lane, part0, (int)nc); break;
        case 1: long_combine<DT, 1, 1>(a, td, key, part0, nc, lane); break;
        case 2: long_combine<DT, 2, 1>(a, td, key, part0, nc, lane); break;
        case 3: long_combine<DT, 4, 1>(a, td, key, part0, nc, lane); break;
        default: long_combine<DT, 4, 2>(a, td, key, part0, nc, lane); break;
    }
}

__global__ void __launch_bounds__(256) long_chunks_kernel(ApplyArgs a, Workspace ws, const uint32_t* pos_sorted) {
    a.has_scale = ws.counters[CTR_HAS_SCALE] != 0;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t nchunks = min(*(volatile uint32_t*)&ws.counters[CTR_NCHUNK], (uint32_t)ws.max_chunks);
    const uint32_t nlong = min(*(volatile uint32_t*)&ws.counters[CTR_NLONG], (uint32_t)ws.max_long);
    for (int64_t c = gw; c < nchunks; c += nw) {
        const uint32_t li = __ldg(ws.chunk_run + c);
        if (li >= nlong) continue;
        const uint32_t u = __ldg(ws.long_runs + 4 * li), base = __ldg(ws.long_runs + 4 * li + 1),
                       nc = __ldg(ws.long_runs + 4 * li + 2);
        const uint32_t j = (uint32_t)c - base;
        const uint32_t key = __ldg(ws.uniq + u);
        const uint32_t r0 = __ldg(ws.runstart + u), r1 = tmin<uint32_t>(__ldg(ws.runstart + u + 1), (uint32_t)a.N);
        const uint32_t s0 = r0 + j * kLongRun, s1 = tmin<uint32_t>(s0 + (uint32_t)kLongRun, r1);
        const int t = table_of(a.tabs, a.T, key);
        const TableDesc td = a.tabs[t];
        switch (td.dtype) {
            case DT_F32: long_dispatch<DT_F32>(a, ws, pos_sorted, td, t, key, s0, s1, (uint32_t)c, li, base, nc, lane); break;
            case DT_F16: long_dispatch<DT_F16>(a, ws, pos_sorted, td, t, key, s0, s1, (uint32_t)c, li, base, nc, lane); break;
            default: long_dispatch<DT_BF16>(a, ws, pos_sorted, td, t, key, s0, s1, (uint32_t)c, li, base, nc, lane); break;
        }
    }
}

cudaError_t launch_apply(const ApplyArgs& a, const Workspace& ws, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    const uint32_t* pos_sorted = ws.vals[ws.sorted_buf];
    const unsigned grid = (unsigned)(a.num_sms * 8);
    short_runs_kernel<<<grid, 256, 0, s>>>(a, ws, pos_sorted);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    long_chunks_kernel<<<grid, 256, 0, s>>>(a, ws, pos_sorted);
    return cudaGetLastError();
}

}  // namespace tbe
