// Dense backward of the small histogram tables (kimbodo "What Happened":
// eligible small tables take a histogram path; backward groups updates by
// (table, row) so each row gets one optimizer update).
//
// A histogram table has at most 1024 rows, and its lookups are the
// contiguous position range [tpos[t], tpos[t+1]) (table-major batch), so its
// gradient  g_r = sum over lookups i with idx_i = r of s_i * G[bag_i, Doff :
// Doff + D]  fits in shared memory and needs no sort:
//
//  dense_accum_kernel: a CTA owns (table, slice of 32*CPL columns, one of S
//    consecutive parts of the table's lookups).  The part's (row, bag, scale)
//    are staged in shared memory a chunk at a time; warp w owns the rows
//    r = w (mod 16) and walks the chunk in position order, adding s * G[bag,
//    c0 + lane + 32*j] to its rows' sums (a gradient row is loaded once per
//    bag change).  Each row is summed by one warp in lookup order, so the
//    result does not depend on scheduling.  The CTA writes its sums to its
//    own slice of the gradient buffer; lookup counts per row are added with
//    integer atomics.
//  dense_update_kernel: one warp per row of every dense table; a row that
//    some lookup touched adds its S partial sums in order, gets its optimizer
//    step (the same SGD / row-wise Adagrad arithmetic as the sorted path) and
//    is stored once.
#include "tbe_internal.cuh"

namespace tbe {

constexpr int kDenseThreads = 512;
constexpr int kDenseWarps = kDenseThreads / 32;
constexpr int kDenseChunk = 2048;  // lookups staged at a time

__host__ __device__ inline int dense_cpl(int64_t max_rows) { return max_rows <= 512 ? 2 : 1; }

__global__ void __launch_bounds__(kDenseThreads) dense_accum_kernel(DenseArgs a, Workspace ws, int cpl,
                                                                    int slices_max) {
    extern __shared__ float s_acc[];  // [rows][32 * cpl], then uint32 counts [rows]
    __shared__ uint16_t s_row[kDenseChunk];
    __shared__ int32_t s_bag[kDenseChunk];
    __shared__ float s_sc[kDenseChunk];
    const int splits = a.splits;
    const int per_table = slices_max * splits;
    const int k = blockIdx.x / per_table;
    const int rem = blockIdx.x % per_table;
    const int cs = rem / splits, sp = rem % splits;
    const int t = a.tables[k];
    const TableDesc td = a.tabs[t];
    const int R = (int)td.rows, D = td.dim;
    const int width = 32 * cpl;
    const int c0 = cs * width;
    if (c0 >= D) return;  // no columns in this slice (whole CTA)
    uint32_t* s_cnt = reinterpret_cast<uint32_t*>(s_acc + (size_t)R * width);
    const bool count = cs == 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < R * width; i += kDenseThreads) s_acc[i] = 0.f;
    if (count)
        for (int i = tid; i < R; i += kDenseThreads) s_cnt[i] = 0;
    // this CTA's part of the table's lookups
    const uint32_t P0 = __ldg(ws.tpos + t);
    const uint32_t P1 = tmax<uint32_t>(__ldg(ws.tpos + t + 1), P0);
    const uint32_t len = P1 - P0;
    const uint32_t q0 = P0 + (uint32_t)(((uint64_t)len * sp) / splits);
    const uint32_t q1 = P0 + (uint32_t)(((uint64_t)len * (sp + 1)) / splits);
    const uint32_t tB = (uint32_t)t * (uint32_t)a.B;
    const bool has_scale = ws.counters[CTR_HAS_SCALE] != 0;
    const float* gcol = a.grad + td.doff + c0 + lane;

    for (uint32_t base = q0; base < q1; base += kDenseChunk) {
        const int n = (int)tmin<uint32_t>((uint32_t)kDenseChunk, q1 - base);
        __syncthreads();  // the previous chunk is consumed (and the sums zeroed)
        for (int i = tid; i < n; i += kDenseThreads) {
            const uint32_t p = base + (uint32_t)i;
            int r = __ldg(ws.hrow + p);
            const uint32_t bag = __ldg(ws.bag + p);
            const int b = (bag >= tB && bag - tB < (uint32_t)a.B) ? (int)(bag - tB) : -1;
            if (r >= R || b < 0) r = 0xffff;  // skipped lookup
            s_row[i] = (uint16_t)r;
            s_bag[i] = b;
            s_sc[i] = has_scale ? __ldg(ws.scale + p) : 1.f;
            if (count && r < R) atomicAdd(&s_cnt[r], 1u);
        }
        __syncthreads();
        int cur = -1;
        float g[2] = {0.f, 0.f};
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            const int r = i < n ? (int)s_row[i] : 0xffff;
            uint32_t mine = __ballot_sync(0xffffffffu, r < R && (r % kDenseWarps) == warp);
            while (mine) {  // this warp's rows, in position order
                const int j = __ffs(mine) - 1;
                mine &= mine - 1;
                const int rj = __shfl_sync(0xffffffffu, r, j);
                const int bj = s_bag[i0 + j];
                const float sj = s_sc[i0 + j];
                if (bj != cur) {  // uniform
                    cur = bj;
                    const float* grow = gcol + (int64_t)bj * a.total_d;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        if (q < cpl) g[q] = (c0 + lane + 32 * q < D) ? __ldg(grow + 32 * q) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if (q < cpl) s_acc[rj * width + lane + 32 * q] = fmaf(sj, g[q], s_acc[rj * width + lane + 32 * q]);
            }
        }
    }
    __syncthreads();
    // this part's sums to its own slice of the gradient buffer; counts added
    float* dg = ws.dgrad + (size_t)sp * a.total_floats + a.goff[k];
    for (int i = tid; i < R * width; i += kDenseThreads) {
        const int rr = i / width, c = c0 + i % width;
        if (c < D) dg[(int64_t)rr * D + c] = s_acc[i];
    }
    if (count) {
        uint32_t* dc = ws.dcount + a.roff[k];
        for (int i = tid; i < R; i += kDenseThreads)
            if (s_cnt[i]) atomicAdd(dc + i, s_cnt[i]);
    }
}

// The row's gradient column c: its parts added in order.
__device__ __forceinline__ float dense_grad(const DenseArgs& a, const float* g, int c) {
    float v = g[c];
    for (int s = 1; s < a.splits; ++s) v += g[(size_t)s * a.total_floats + c];
    return v;
}

template <int DT>
__device__ __forceinline__ void dense_update_row(const DenseArgs& a, const TableDesc& td, const float* g, int64_t r,
                                                 int lane) {
    const int D = td.dim;
    float gv[8];  // this lane's columns lane + 32*j (D <= 256)
#pragma unroll
    for (int j = 0; j < 8; ++j) gv[j] = lane + 32 * j < D ? dense_grad(a, g, lane + 32 * j) : 0.f;
    float m = 0.f, denom = 1.f;
    if (a.opt == 2) {
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) sq = fmaf(gv[j], gv[j], sq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        m = a.state[td.rowbase + r] + __fdiv_rn(sq, (float)D);
        denom = sqrtf(m) + a.eps;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = lane + 32 * j;
        if (c >= D) continue;
        const float w = load_elem<DT>(td.data, r * D + c);
        const float nw = a.opt == 2 ? w - a.lr * __fdiv_rn(gv[j], denom) : fmaf(-a.lr, gv[j], w);
        store_elem<DT>(td.data, r * D + c, nw);
    }
    if (a.opt == 2 && lane == 0) a.state[td.rowbase + r] = m;
}

__global__ void __launch_bounds__(256) dense_update_kernel(DenseArgs a, Workspace ws) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // one warp per row
    if (gw >= a.total_rows) return;
    int lo = 0, hi = a.n - 1;  // dense table of row gw: last k with roff[k] <= gw
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.roff[mid] <= gw)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int64_t r = gw - a.roff[lo];
    if (ws.dcount[a.roff[lo] + r] == 0) return;  // untouched: never written
    const TableDesc td = a.tabs[a.tables[lo]];
    const float* g = ws.dgrad + a.goff[lo] + r * td.dim;  // part 0; part s at + s * total_floats
    if (td.dtype == DT_F16)
        dense_update_row<DT_F16>(a, td, g, r, lane);
    else if (td.dtype == DT_BF16)
        dense_update_row<DT_BF16>(a, td, g, r, lane);
    else
        dense_update_row<DT_F32>(a, td, g, r, lane);
}

// Clears the row counts, sums, updates (all on stream s).
cudaError_t launch_dense(const DenseArgs& a, const Workspace& ws, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(ws.dcount, 0, sizeof(uint32_t) * (size_t)a.total_rows, s);
    if (e != cudaSuccess) return e;
    const int cpl = dense_cpl(a.max_rows);
    const int width = 32 * cpl;
    const int slices_max = (a.max_dim + width - 1) / width;
    const size_t smem = (size_t)a.max_rows * width * sizeof(float) + (size_t)a.max_rows * sizeof(uint32_t);
    static size_t configured = 0;  // largest dynamic shared memory set so far
    if (smem > configured) {
        e = cudaFuncSetAttribute(dense_accum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    const unsigned grid = (unsigned)(a.n * slices_max * a.splits);
    dense_accum_kernel<<<grid, kDenseThreads, smem, s>>>(a, ws, cpl, slices_max);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned ublocks = (unsigned)((a.total_rows * 32 + 255) / 256);
    dense_update_kernel<<<ublocks, 256, 0, s>>>(a, ws);
    return cudaGetLastError();
}

}  // namespace tbe
