// Dense backward of the small histogram tables (kimbodo "What Happened":
// eligible small tables take a histogram and tensor-core path; backward
// groups updates by (table, row) so each row gets one optimizer update).
//
// A histogram table has at most 1024 rows, so its whole gradient is one
// dense product:  dW = H^T . G_t, with H[b, r] = the sum of the scales s_i
// of bag b's lookups of row r and G_t the table's columns of the upstream
// gradient.  Its lookups need no sort:
//
//  dense_mma_kernel: a CTA owns (table, up to four 128-row M tiles, one of S
//    consecutive bag ranges).  For every 32 bags it builds H^T (rows x bags)
//    and G_t (columns x bags) in shared memory in the no-swizzle K-major
//    core-matrix layout and issues tcgen05.mma (kind::f16, bf16 operands,
//    fp32 accumulator in tensor memory, M = 128, N = dim, K = 16).  For fp32
//    accuracy both operands are split into three bf16 terms,
//    x = x0 + x1 + x2 (24 significant bits), and the six products with
//    i + j <= 2 are accumulated.  H^T is built without races: warp w owns
//    bags w and w + 16 of the tile and walks their lookups in order,
//    merging
//    repeated rows (ballot match) so every entry has one writer; results
//    do not depend on scheduling.  Every kDenseFlush bag tiles, and after its
//    last one, the CTA reads the accumulator back (tcgen05.ld) and adds it to
//    its own slice of the gradient buffer (fp32, fixed order), then restarts
//    the accumulator; at the end it adds its lookup counts per row (integer
//    atomics).
//  dense_update_kernel: one warp per row of every dense table; a row that
//    some lookup touched adds its S partial sums in order, gets its optimizer
//    step (the same SGD / row-wise Adagrad arithmetic as the sorted path) and
//    is stored once.
#include "tbe_internal.cuh"
#include "tcgen05.cuh"

namespace tbe {

constexpr int kDenseThreads = 512;
constexpr int kDenseWarps = kDenseThreads / 32;
constexpr int kDenseKT = 32;      // bags per tile (two MMA K steps)
constexpr int kDenseSplit = 3;    // bf16 terms per operand
constexpr int kDenseMaxMp = 512;  // rows per CTA (four 128-row M tiles)
// Bag tiles summed in tensor memory before the partial sum is added to the
// CTA's gradient slice in fp32 (round to nearest).  The tensor cores' own
// accumulation rounds each step against the magnitude of the running sum;
// restarting it every few tiles keeps that sum, and so the error, small.
constexpr int kDenseFlush = 32;

// bf16 bits of x rounded to nearest even, and the value they stand for.
__device__ __forceinline__ uint16_t to_bf16(float x, float& back) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    back = __bfloat162float(h);
    return __bfloat16_as_ushort(h);
}

// x as three bf16 terms x0 + x1 + x2.
__device__ __forceinline__ void split3(float x, uint16_t (&t)[kDenseSplit]) {
    float b;
    t[0] = to_bf16(x, b);
    x -= b;
    t[1] = to_bf16(x, b);
    x -= b;
    t[2] = to_bf16(x, b);
}

__device__ __forceinline__ float bf16_value(uint16_t bits) { return __uint_as_float((uint32_t)bits << 16); }

// Shared-memory plan of one CTA for Mp rows and dim D (bytes).
__host__ __device__ inline size_t dense_a_bytes(int Mp) { return (size_t)Mp * kDenseKT * 2; }
__host__ __device__ inline size_t dense_b_bytes(int D) { return (size_t)D * kDenseKT * 2; }
__host__ __device__ inline size_t dense_smem_bytes(int Mp, int D) {
    return kDenseSplit * (dense_a_bytes(Mp) + dense_b_bytes(D)) + sizeof(uint32_t) * (size_t)Mp;
}

// 128-row M tiles per CTA for dim D: the accumulator takes D tensor-memory
// columns per tile, 512 columns in all.
__host__ __device__ inline int dense_mtiles(int D) {
    const int by_tmem = 512 / D;
    return by_tmem < kDenseMaxMp / 128 ? by_tmem : kDenseMaxMp / 128;
}

__host__ __device__ inline uint32_t dense_tmem_cols(int n) {
    return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

__global__ void __launch_bounds__(kDenseThreads, 1) dense_mma_kernel(DenseArgs a, Workspace ws, int groups_max) {
    extern __shared__ __align__(1024) unsigned char dsm[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    constexpr int kMaxMma = (kDenseMaxMp / 128) * (kDenseKT / 16) * 6;
    __shared__ uint64_t s_adesc[kMaxMma], s_bdesc[kMaxMma];
    __shared__ uint32_t s_dcol[kMaxMma];
    __shared__ bool s_init[kMaxMma];
    const int splits = a.splits;
    const int per_table = groups_max * splits;
    const int k = blockIdx.x / per_table;
    const int rem = blockIdx.x % per_table;
    const int mg = rem / splits, sp = rem % splits;
    const int t = a.tables[k];
    const TableDesc td = a.tabs[t];
    const int R = (int)td.rows, D = td.dim;
    const int mt_per = dense_mtiles(D);
    const int row0 = mg * mt_per * 128;
    if (row0 >= R) return;  // no rows in this group (whole CTA)
    const int rows_here = tmin<int>(R - row0, mt_per * 128);
    const int mtiles = (rows_here + 127) / 128;
    const int Mp = mtiles * 128;  // rows of this CTA's A tiles
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    unsigned char* As = dsm;                                    // [split][Mp x KT] bf16
    unsigned char* Bs = dsm + kDenseSplit * dense_a_bytes(Mp);  // [split][D x KT] bf16
    uint32_t* s_cnt = reinterpret_cast<uint32_t*>(Bs + kDenseSplit * dense_b_bytes(D));  // [Mp]
    const uint32_t sbo = (uint32_t)(kDenseKT / 8) * 128u;  // bytes per 8 rows (K-major core matrices)

    // bag range of this part
    const int bk0 = (int)(((int64_t)a.B * sp) / splits);
    const int bk1 = (int)(((int64_t)a.B * (sp + 1)) / splits);
    const uint32_t* boff = ws.dboff + (int64_t)td.dslot * (a.B + 1);
    const bool has_scale = ws.counters[CTR_HAS_SCALE] != 0;
    const bool gvec = a.grad_vec && td.doff % 4 == 0;
    const uint32_t ncols = dense_tmem_cols(mtiles * D);
    if (warp == 0) tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < Mp; i += kDenseThreads) s_cnt[i] = 0;
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = mma_idesc(1, 128, D);  // bf16 x bf16 -> fp32
    const uint32_t abase = smem_u32(As), bbase = smem_u32(Bs);
    // the tile's MMAs: the six products x_i * y_j with i + j <= 2 for every
    // M tile and both K steps (descriptors are the same for every tile)
    const int nmma = mtiles * (kDenseKT / 16) * 6;
    if (tid < nmma) {
        // product pr: terms (pa, pb) = (0,0) (0,1) (1,0) (0,2) (1,1) (2,0), two bits each
        const int pr = tid % 6, ks = (tid / 6) % (kDenseKT / 16), i = tid / (6 * (kDenseKT / 16));
        const int pa = (0x910 >> (2 * pr)) & 3, pb = (0x184 >> (2 * pr)) & 3;
        const uint32_t ad = abase + (uint32_t)(pa * dense_a_bytes(Mp)) + (uint32_t)(i * 16) * sbo + 256u * ks;
        const uint32_t bd = bbase + (uint32_t)(pb * dense_b_bytes(D)) + 256u * ks;
        s_adesc[tid] = smem_desc(ad, 128u, sbo);
        s_bdesc[tid] = smem_desc(bd, 128u, sbo);
        s_dcol[tid] = (uint32_t)(i * D);
        s_init[tid] = ks == 0 && pr == 0;  // the first MMA of each M tile starts the sum
    }
    __syncthreads();
    uint32_t phase = 0;
    bool first = true, timed_out = false, written = false;
    int in_acc = 0;  // bag tiles in the accumulator since the last flush
    float* dg = ws.dgrad + (size_t)sp * a.total_floats + a.goff[k];
    const int lg = warp & 3;  // warp w reads tensor-memory lanes 32*(w%4) .. +31
    // accumulator (or zeros, when it holds no tile) -> this part's gradient
    // slice: stored by the first flush, added by the later ones
    auto flush = [&]() {
        for (int i = 0; i < mtiles; ++i) {
            const int r = row0 + i * 128 + lg * 32 + lane;
            for (int c = (warp >> 2) * 16; c < D; c += (kDenseWarps / 4) * 16) {
                float v[16];
                if (!first) {
                    tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)(i * D + c), v);  // whole warp
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] = 0.f;
                }
                if (r < R) {
                    float4* dst = reinterpret_cast<float4*>(dg + (int64_t)r * D + c);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        if (written) {
                            const float4 p = dst[q];
                            o.x = p.x + o.x;
                            o.y = p.y + o.y;
                            o.z = p.z + o.z;
                            o.w = p.w + o.w;
                        }
                        dst[q] = o;
                    }
                }
            }
        }
        written = true;
        first = true;  // the next tile's first MMAs overwrite the accumulator
        in_acc = 0;
    };

    // Registers holding the next tile's inputs, loaded while the previous
    // tile's MMAs run: gradient vectors (element e = tid + 512*q of the
    // tile's KT x D/4 float4 grid) and, per owned bag, its lookup range and
    // first 32 lookups.
    constexpr int kBagsPerWarp = kDenseKT / kDenseWarps;
    constexpr int kGPre = 2;  // prefetched: dim <= 128 (the rest of a dim-256 tile loads in place)
    float4 gpre[kGPre];
    uint32_t bp[kBagsPerWarp], bq[kBagsPerWarp];
    int rpre[kBagsPerWarp];
    float spre[kBagsPerWarp];
    auto prefetch = [&](int b0) {
        const int nb = tmin<int>(kDenseKT, bk1 - b0);
#pragma unroll
        for (int q = 0; q < kGPre; ++q) {
            const int e = tid + q * kDenseThreads;
            const int j = e / (D / 4), c4 = (e % (D / 4)) * 4;
            gpre[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < kDenseKT * (D / 4) && j < nb) {
                const float* gp = a.grad + (int64_t)(b0 + j) * a.total_d + td.doff + c4;
                if (gvec) {
                    gpre[q] = __ldg(reinterpret_cast<const float4*>(gp));
                } else {
                    gpre[q].x = __ldg(gp);
                    gpre[q].y = __ldg(gp + 1);
                    gpre[q].z = __ldg(gp + 2);
                    gpre[q].w = __ldg(gp + 3);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kBagsPerWarp; ++h) {
            const int j = warp + h * kDenseWarps;
            bp[h] = bq[h] = 0;
            rpre[h] = 0xffff;
            spre[h] = 0.f;
            if (j < nb) {
                bp[h] = __ldg(boff + b0 + j);
                bq[h] = tmax<uint32_t>(__ldg(boff + b0 + j + 1), bp[h]);
                const uint32_t p = bp[h] + lane;
                if (p < bq[h]) {
                    rpre[h] = __ldg(ws.hrow + p);
                    spre[h] = has_scale ? __ldg(ws.scale + p) : 1.f;
                }
            }
        }
    };
    if (bk0 < bk1) prefetch(bk0);

    for (int b0 = bk0; b0 < bk1; b0 += kDenseKT) {
        // clear A (all terms)
        {
            uint4* pa = reinterpret_cast<uint4*>(As);
            const int n16 = (int)(kDenseSplit * dense_a_bytes(Mp) / 16);
            for (int i = tid; i < n16; i += kDenseThreads) pa[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        // B from the prefetched gradient vectors (bags past the range are
        // zeros); element (n = column, k = bag)
        const int nb = tmin<int>(kDenseKT, bk1 - b0);
#pragma unroll
        for (int q = 0; q < kDenseKT * 256 / 4 / kDenseThreads; ++q) {  // dim <= 256
            const int e = tid + q * kDenseThreads;
            if (e >= kDenseKT * (D / 4)) continue;
            const int j = e / (D / 4), c4 = (e % (D / 4)) * 4;
            float4 gv4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q < kGPre) {
                gv4 = gpre[q];
            } else if (j < nb) {
                const float* gp = a.grad + (int64_t)(b0 + j) * a.total_d + td.doff + c4;
                gv4 = make_float4(__ldg(gp), __ldg(gp + 1), __ldg(gp + 2), __ldg(gp + 3));
            }
            const float f[4] = {gv4.x, gv4.y, gv4.z, gv4.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint16_t tt[kDenseSplit];
                split3(f[c], tt);
#pragma unroll
                for (int si = 0; si < kDenseSplit; ++si)
                    *reinterpret_cast<uint16_t*>(Bs + si * dense_b_bytes(D) + core_off(c4 + c, j, sbo)) = tt[si];
            }
        }
        __syncthreads();  // A cleared before the histogram is written
        // H^T: warp w owns bags w and w + 16 of the tile; lookups in order,
        // repeated rows merged so each entry has one writer
#pragma unroll
        for (int h = 0; h < kBagsPerWarp; ++h) {
            const int j = warp + h * kDenseWarps;
            for (uint32_t x = bp[h]; x < bq[h]; x += 32) {
                int r;
                float sc;
                if (x == bp[h]) {  // the prefetched first 32 lookups
                    r = rpre[h];
                    sc = spre[h];
                } else {
                    const uint32_t p = x + lane;
                    r = 0xffff;
                    sc = 0.f;
                    if (p < bq[h]) {
                        r = __ldg(ws.hrow + p);
                        sc = has_scale ? __ldg(ws.scale + p) : 1.f;
                    }
                }
                const int m = r - row0;
                const bool mine = r < R && m >= 0 && m < Mp;
                const uint32_t lab = mine ? (uint32_t)m : 2047u;  // rows of other groups / skipped: one label
                const uint32_t peers = match_label<11>(lab);
                // the group's scales, added in lane order (groups of one: the scale)
                float tot = sc;
                if (__any_sync(0xffffffffu, mine && __popc(peers) > 1)) {
                    tot = 0.f;
                    for (int l = 0; l < 32; ++l) {
                        const float v = __shfl_sync(0xffffffffu, sc, l);
                        if ((peers >> l) & 1u) tot += v;
                    }
                }
                if (mine && (peers & ((1u << lane) - 1u)) == 0) {
                    // entry (m, j): value so far (earlier lookups of the bag) + tot
                    float prev = 0.f;
                    uint16_t tt[kDenseSplit];
                    if (x != bp[h]) {
#pragma unroll
                        for (int si = 0; si < kDenseSplit; ++si)
                            prev += bf16_value(
                                *reinterpret_cast<uint16_t*>(As + si * dense_a_bytes(Mp) + core_off(m, j, sbo)));
                    }
                    split3(prev + tot, tt);
#pragma unroll
                    for (int si = 0; si < kDenseSplit; ++si)
                        *reinterpret_cast<uint16_t*>(As + si * dense_a_bytes(Mp) + core_off(m, j, sbo)) = tt[si];
                    atomicAdd(&s_cnt[m], (uint32_t)__popc(peers));
                }
            }
        }
        fence_proxy_async_smem();  // generic-proxy writes of A and B -> tensor cores
        tcgen05_before_sync();
        __syncthreads();
        tcgen05_after_sync();
        if (tid == 0) {
            for (int q = 0; q < nmma; ++q)
                mma_f16(tmem + s_dcol[q], s_adesc[q], s_bdesc[q], idesc, (first && s_init[q]) ? 0u : 1u);
            mma_commit(&s_bar);
        }
        first = false;
        // the next tile's inputs load while the MMAs run
        if (b0 + kDenseKT < bk1) prefetch(b0 + kDenseKT);
        // every thread waits; the block agrees on the outcome
        const bool ok = mbar_wait(&s_bar, phase);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        phase ^= 1u;
        tcgen05_after_sync();
        // each thread reads and writes only its own accumulator rows and
        // columns, and the sync before the next MMAs orders the reads first
        if (++in_acc == kDenseFlush || b0 + kDenseKT >= bk1) flush();
    }
    if (!timed_out) {
        if (!written) flush();  // a part with no bags stores zeros
        uint32_t* dc = ws.dcount + a.roff[k] + row0;
        for (int i = tid; i < rows_here; i += kDenseThreads)
            if (s_cnt[i]) atomicAdd(dc + i, s_cnt[i]);
    } else {
        if (tid == 0) atomicOr(&a.blk->error, ERR_TIMEOUT);
        mbar_wait(&s_bar, phase);  // a second bounded wait for the MMAs in flight
    }
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    if (warp == 0) tmem_dealloc(tmem, ncols);
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
    // the largest plan over dims up to max_dim and rows up to max_rows
    size_t smem = 0;
    int groups_max = 1;
    for (int D = 16; D <= a.max_dim; D += 16) {
        const int Mg = dense_mtiles(D) * 128;
        const int Mp = tmin<int>(Mg, (a.max_rows + 127) / 128 * 128);
        smem = tmax<size_t>(smem, dense_smem_bytes(Mp, D));
        groups_max = tmax<int>(groups_max, (a.max_rows + Mg - 1) / Mg);
    }
    static size_t configured = 0;  // largest dynamic shared memory set so far
    if (smem > configured) {
        e = cudaFuncSetAttribute(dense_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    const unsigned grid = (unsigned)(a.n * groups_max * a.splits);
    dense_mma_kernel<<<grid, kDenseThreads, smem, s>>>(a, ws, groups_max);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned ublocks = (unsigned)((a.total_rows * 32 + 255) / 256);
    dense_update_kernel<<<ublocks, 256, 0, s>>>(a, ws);
    return cudaGetLastError();
}

}  // namespace tbe
