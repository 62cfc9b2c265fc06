// Small-table forward path on the tensor cores (kimbodo "What Happened":
// eligible small tables use a histogram and tensor-core path).
//
// For a table with few rows, pooling is a dense product: with
//   H[b, r] = sum over the lookups i of bag b with idx_i = r of s_i
// (s_i = per-sample weight, times 1/L for mean pooling), the pooled rows are
//   out[b, Doff : Doff + D] = H[b, :] . W   (H: B x R, W: R x D).
// A CTA of 16 warps keeps W^T (D x R, zero-padded in R to Kp) in shared
// memory and, for each tile of 128 bags, builds H (128 x Kp) in shared memory
// with 16-bit atomic adds, issues Kp/16 tcgen05.mma (kind::f16, M=128, N=D,
// K=16, fp32 accumulation in tensor memory), waits on an mbarrier that
// tcgen05.commit arrives on, and reads the accumulator back with tcgen05.ld
// (warp w may read tensor-memory lanes 32*(w%4) .. +31, i.e. bags 32*(w%4) ..
// +31 of the tile; the four warps sharing a lane quarter split the columns
// in 16-column steps).  H and W^T use the no-swizzle K-major layout of 8x16-byte core
// matrices: element (m, k) of an operand with row stride SBO bytes per 8
// rows sits at (m/8)*SBO + (k/8)*128 + (m%8)*16 + (k%8)*2.
//
// Both operands are fp16 (the tensor cores take A and B in one type): fp16
// tables as they are, bf16 tables converted (exact within fp16's normal
// range), H entries as fp16 sums of lookup scales.  Products and sums are
// fp32.  A table value that does not fit fp16 sends the table to an fp32
// gather; an H sum beyond 65504 (seen as non-finite outputs of its bag)
// sends its tile there.
#include "tbe_internal.cuh"
#include "tcgen05.cuh"

namespace tbe {

constexpr int kHistM = 128;          // bags per tile (MMA M)
constexpr int kHistThreads = 512;    // 16 warps; warp w reads tensor-memory lanes 32*(w%4)..
constexpr int kHistTilesPerCta = 8;  // bag tiles per CTA (W^T is loaded once)

constexpr float kHalfMax = 65504.f;
constexpr int kHistBagofCap = 8192;  // positions of a tile whose bag is tabulated in shared memory
constexpr int kHistInFlight = 12;    // lookups per thread whose index and weight loads are in flight together

// fp16 add to a shared-memory half (a shared-space reduction: nothing waits
// for its result).
__device__ __forceinline__ void red_add_half_shared(unsigned char* p, __half v) {
    asm volatile("red.shared.add.noftz.f16 [%0], %1;" ::"r"(smem_u32(p)), "h"(__half_as_ushort(v)) : "memory");
}

// Fallback for a tile whose values do not fit the fp16 operands: warp per
// bag, lanes over columns, fp32 accumulation straight from the table.
template <int DT, typename IDX>
__device__ void hist_tile_gather(const FwdArgs& a, const TableDesc& td, int t, int b0, int nb, int warp,
                                 int lane, bool& oob) {
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const int D = td.dim;
    for (int m = warp; m < nb; m += kHistThreads / 32) {
        const int b = b0 + m;
        const int64_t bag = (int64_t)t * a.B + b;
        int64_t start = ld_index(off, bag), end = ld_index(off, bag + 1);
        if (start < 0 || end < start || end > a.N) start = end = 0;
        float* orow = a.out + (int64_t)b * a.total_d + td.doff;
        for (int c0 = 0; c0 < D; c0 += 256) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int64_t p = start; p < end; ++p) {
                const int64_t x = ld_index(ind, p);
                if (x < 0 || x >= td.rows) {
                    oob = true;
                    continue;
                }
                const float s = a.weights ? __ldg(a.weights + p) : 1.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = c0 + lane + 32 * j;
                    if (c < D) acc[j] = fmaf(s, load_elem<DT>(td.data, x * D + c), acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = c0 + lane + 32 * j;
                if (c < D) orow[c] = (a.mean && end > start) ? __fdiv_rn(acc[j], (float)(end - start)) : acc[j];
            }
        }
    }
}

template <int DT, typename IDX>
__global__ void __launch_bounds__(kHistThreads, 1) hist_kernel(FwdArgs a, const int32_t* hist_tables,
                                                             int ctas_per_table) {
    chain_wait();  // returns at once unless launched chained
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_wovf;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = hist_tables[blockIdx.x / ctas_per_table];
    const int cta = blockIdx.x % ctas_per_table;
    const TableDesc td = a.tabs[t];
    const int R = (int)td.rows, D = td.dim;
    const int Kp = (R + 15) & ~15;
    const uint32_t sbo = (uint32_t)(Kp / 8) * 128u;  // bytes per 8 rows of H (bags) and of W^T (columns)
    unsigned char* Hs = smem_raw;
    unsigned char* Ws = smem_raw + (size_t)kHistM * Kp * 2;
    // the CTA's bag offsets (clamped to [-1, N + 1]: positions are below 2^30)
    int32_t* s_off = reinterpret_cast<int32_t*>(Ws + (size_t)D * Kp * 2);
    // bag within the tile of each of the tile's first kHistBagofCap positions
    uint8_t* s_bagof = reinterpret_cast<uint8_t*>(s_off + kHistTilesPerCta * kHistM + 1);
    const int ntiles = (a.B + kHistM - 1) / kHistM;
    const int tile0 = cta * kHistTilesPerCta;
    if (tile0 >= ntiles) return;  // whole CTA leaves before allocating anything
    const int tile1 = tile0 + kHistTilesPerCta < ntiles ? tile0 + kHistTilesPerCta : ntiles;
    const int bag_lo = tile0 * kHistM;
    const int bag_hi = tile1 * kHistM < a.B ? tile1 * kHistM : a.B;
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const uint32_t ncols = D <= 32 ? 32u : (D <= 64 ? 64u : (D <= 128 ? 128u : 256u));
    bool oob = false, bad_off = false, timed_out = false;

    if (warp == 0) tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        s_wovf = 0;
        mbar_init(&s_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // bag offsets of the CTA's tiles
    for (int i = tid; i <= bag_hi - bag_lo; i += kHistThreads)
        s_off[i] = (int32_t)tmin<int64_t>(tmax<int64_t>(ld_index(off, (int64_t)t * a.B + bag_lo + i), -1), a.N + 1);
    // W^T as fp16: element (n, k) = W[k][n], zero for k >= R
    const unsigned short* W = reinterpret_cast<const unsigned short*>(td.data);
    int ovf = 0;
    for (int e = tid; e < Kp * (D / 8); e += kHistThreads) {
        const int k = e / (D / 8), n8 = (e % (D / 8)) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k < R) v = __ldg(reinterpret_cast<const uint4*>(W + (int64_t)k * D + n8));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t bits = (w4[j >> 1] >> (16 * (j & 1))) & 0xffffu;
            if constexpr (DT == DT_BF16) {
                // bf16 -> fp16 is exact inside fp16's normal range; a finite
                // value beyond it would become inf: take the fallback
                const float f = bf16_bits_to_float(bits);
                if (fabsf(f) > kHalfMax && isfinite(f)) ovf = 1;
                bits = __half_as_ushort(__float2half_rn(f));
            }
            *reinterpret_cast<unsigned short*>(Ws + core_off(n8 + j, k, sbo)) = (unsigned short)bits;
        }
    }
    if (ovf) s_wovf = 1;
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = mma_idesc(0, kHistM, D);  // fp16 x fp16 -> fp32
    const uint64_t hdesc0 = smem_desc(smem_u32(Hs), 128u, sbo), wdesc0 = smem_desc(smem_u32(Ws), 128u, sbo);
    const bool mean = a.mean != 0;
    const bool wovf = s_wovf != 0;
    uint32_t phase = 0;

    for (int tile = tile0; tile < tile1; ++tile) {
        const int b0 = tile * kHistM;
        const int nb = b0 + kHistM < a.B ? kHistM : a.B - b0;
        const int32_t* toff = s_off + (b0 - bag_lo);  // toff[0..nb]
        if (wovf) {  // the table does not fit fp16: every tile by fp32 gather
            hist_tile_gather<DT, IDX>(a, td, t, b0, nb, warp, lane, oob);
            continue;
        }
        // zero H; tabulate the bag of each position (four threads per bag)
        for (int e = tid; e < kHistM * Kp * 2 / 16; e += kHistThreads)
            reinterpret_cast<uint4*>(Hs)[e] = make_uint4(0u, 0u, 0u, 0u);
        const int64_t P0 = toff[0], P1 = toff[nb];
        {
            const int m = tid >> 2, sub = tid & 3;
            bool bad = false;
            if (m < nb) {
                bad = toff[m + 1] < toff[m];
                const int64_t s0 = tmax<int64_t>(toff[m], P0), s1 = tmin<int64_t>(toff[m + 1], P0 + kHistBagofCap);
                for (int64_t q = s0 + sub; q < s1; q += 4) s_bagof[q - P0] = (uint8_t)m;
            }
            // offsets that do not rise monotonically: every position searches
            if (__syncthreads_or(bad)) bad_off = true;
        }
        const bool tab_ok = !bad_off;
        // histogram of the tile: its lookups are the contiguous range
        // [toff[0], toff[nb]); per block of 512 positions, thread t takes
        // position (t % 8) * 64 + t / 8, so a warp's 32 lookups come from 8
        // runs of 4 (8 bags, mostly: their H entries spread over the banks)
        // while its index loads stay 8 whole sectors; kHistInFlight in flight
        const bool range_ok = P0 >= 0 && P1 >= P0 && P1 <= a.N;
        if (!range_ok) bad_off = true;
        const int perm = (tid & 7) * 64 + (tid >> 3);
        for (int64_t base = P0; range_ok && base < P1; base += kHistInFlight * kHistThreads) {
            const int64_t pb = base + perm;
            int64_t x[kHistInFlight];
            float w[kHistInFlight];
#pragma unroll
            for (int u = 0; u < kHistInFlight; ++u) {
                const int64_t p = pb + (int64_t)u * kHistThreads;
                x[u] = -1;
                w[u] = 1.f;
                if (p < P1) {
                    x[u] = ld_index(ind, p);
                    if (a.weights) w[u] = __ldg(a.weights + p);
                }
            }
#pragma unroll
            for (int u = 0; u < kHistInFlight; ++u) {
                const int64_t p = pb + (int64_t)u * kHistThreads;
                if (p >= P1) continue;
                // bag of position p: tabulated, else (a long tile, or offsets
                // that do not rise monotonically) the last m with toff[m] <= p
                int lo = p - P0 < kHistBagofCap ? s_bagof[p - P0] : 0;
                if (!(tab_ok && p - P0 < kHistBagofCap)) {
                    lo = 0;
                    int hi = nb - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (toff[mid] <= p)
                            lo = mid;
                        else
                            hi = mid - 1;
                    }
                }
                const int64_t L = toff[lo + 1] - toff[lo];
                if (L <= 0) {  // malformed offsets: p belongs to no bag
                    bad_off = true;
                    continue;
                }
                if (x[u] < 0 || x[u] >= R) {
                    oob = true;
                    continue;
                }
                float s = w[u];
                if (mean) s = __fdiv_rn(s, (float)L);
                red_add_half_shared(Hs + core_off(lo, (int)x[u], sbo), __float2half_rn(s));
            }
        }
        fence_proxy_async_smem();  // generic-proxy writes of H -> tensor cores
        tcgen05_before_sync();
        __syncthreads();
        tcgen05_after_sync();
        if (tid == 0) {
            // K step j: both descriptors' start address field (address >> 4)
            // moves by 256 bytes (the field does not carry: addresses < 2^18)
            for (int j = 0; j < Kp / 16; ++j)
                mma_f16(tmem, hdesc0 + (uint64_t)(16 * j), wdesc0 + (uint64_t)(16 * j), idesc, j > 0 ? 1u : 0u);
            mma_commit(&s_bar);
        }
        // every thread waits; the block agrees on the outcome so all threads
        // take the same path through the barriers below
        const bool ok = mbar_wait(&s_bar, phase);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        phase ^= 1u;
        tcgen05_after_sync();
        // accumulator -> output: warp w reads tensor-memory lanes 32*(w%4)..
        // (bags of the tile) and the 16-column chunks c = w/4, w/4 + 4, ...
        const int lg = warp & 3;
        const int b = b0 + lg * 32 + lane;
        float* orow = a.out + (int64_t)b * a.total_d + td.doff;
        bool nonfinite = false;
        for (int c = (warp >> 2) * 16; c < D; c += (kHistThreads / 128) * 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(lg * 32) << 16) + (uint32_t)c, v);  // whole warp, aligned
            if (b < a.B) {
#pragma unroll
                for (int q = 0; q < 16; ++q) nonfinite |= !isfinite(v[q]);
                if (a.vec_out) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<float4*>(orow + c)[q] =
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) orow[c + q] = v[q];
                }
            }
        }
        // an H entry past fp16's range makes its bag's outputs inf or NaN
        // (so do inf/NaN inputs): such a tile is redone by the fp32 gather
        if (__syncthreads_or(nonfinite)) hist_tile_gather<DT, IDX>(a, td, t, b0, nb, warp, lane, oob);
        tcgen05_before_sync();
        __syncthreads();  // accumulator read and H consumed before the next tile
        tcgen05_after_sync();
    }
    if (timed_out) {
        if (tid == 0) atomicOr(&a.blk->error, ERR_TIMEOUT);
        mbar_wait(&s_bar, phase);  // a second bounded wait for the MMAs in flight
    }
    if (oob) atomicOr(&a.blk->error, ERR_OOB);
    if (bad_off) atomicOr(&a.blk->error, ERR_OFFSETS);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

// Shared memory of the histogram kernel for a table of R rows and dim D.
size_t hist_smem_bytes(int64_t R, int D) {
    const int64_t Kp = (R + 15) & ~int64_t(15);
    return (size_t)(kHistM + D) * Kp * 2 + sizeof(int32_t) * (kHistTilesPerCta * kHistM + 1) + kHistBagofCap;
}

int hist_ctas_per_table(int B) {
    const int ntiles = (B + kHistM - 1) / kHistM;
    return (ntiles + kHistTilesPerCta - 1) / kHistTilesPerCta;
}

template <int DT, typename IDX>
static cudaError_t launch_hist_t(const FwdArgs& a, const int32_t* hist_tables, int nhist, size_t smem,
                                 cudaStream_t s) {
    static size_t configured = 0;  // largest dynamic shared memory set so far
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(hist_kernel<DT, IDX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    const int per = hist_ctas_per_table(a.B);
    // the forward's long-bag kernel (or the other dtype's launch) runs just before
    return launch_chained_smem(hist_kernel<DT, IDX>, dim3((unsigned)(nhist * per)), dim3(kHistThreads), smem, s, a,
                               hist_tables, per);
}

// One launch per table dtype (f16, bf16) that has histogram tables.
cudaError_t launch_hist(const FwdArgs& a, const int32_t* hist_tables_f16, int n_f16, size_t smem_f16,
                        const int32_t* hist_tables_bf16, int n_bf16, size_t smem_bf16, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (n_f16 > 0)
        e = a.idx64 ? launch_hist_t<DT_F16, int64_t>(a, hist_tables_f16, n_f16, smem_f16, s)
                    : launch_hist_t<DT_F16, int32_t>(a, hist_tables_f16, n_f16, smem_f16, s);
    if (e == cudaSuccess && n_bf16 > 0)
        e = a.idx64 ? launch_hist_t<DT_BF16, int64_t>(a, hist_tables_bf16, n_bf16, smem_bf16, s)
                    : launch_hist_t<DT_BF16, int32_t>(a, hist_tables_bf16, n_bf16, smem_bf16, s);
    return e;
}

}  // namespace tbe
