// Small-table forward path on the tensor cores (kimbodo "What Happened":
// eligible small tables use a histogram and tensor-core path, with
// higher-precision accumulation).
//
// For a table with few rows, pooling is a dense product: with
//   H[b, r] = sum over the lookups i of bag b with idx_i = r of s_i
// (s_i = per-sample weight, times 1/L for mean pooling), the pooled rows are
//   out[b, Doff : Doff + D] = H[b, :] . W   (H: B x R, W: R x D).
//
// Precision.  Every H entry is summed in fp32 and handed to the tensor cores
// as two fp16 terms, hi = fp16(x) and lo = fp16(x - hi), so it keeps about 22
// significant bits.  fp16 has a narrow exponent range, so each bag's scales
// are multiplied by a power of two 2^e_b chosen from S_b = sum |s_i| (every
// |H[b, r]| <= S_b): S_b * 2^e_b lies in [2^14, 2^15), far from fp16's
// overflow, and an entry loses relative precision only where it is below
// S_b * 2^-28.  fp16 tables enter as they are; a bf16 table is multiplied by
// a power of two 2^f chosen from its largest magnitude the same way, which is
// exact for every value within 2^29 of that magnitude.  The products and sums
// are fp32 in tensor memory; the epilogue adds the hi and lo products and
// multiplies by 2^-(e_b + f).
//
// Schedule.  A tile is 64 bags.  The MMA's A operand (M = 128 rows) holds hi
// and lo of the tile's 64 bags; the 8-row group g of A belongs to warp g of
// the CTA: its rows 0-3 are hi of the warp's four bags, rows 4-7 their lo.  Each warp
// walks its four bags' lookups (contiguous positions) 32 at a time; lanes
// with the same (bag, row) are grouped with a warp match, the group's scales
// are added in lane order, and one lane adds the group sum into the H entry
// (read hi + lo, add, split again).  A warp owns its rows of A, so no two
// warps touch one entry: no atomics, and the result does not depend on
// scheduling.  Per tile: one elected thread issues Kp/16 tcgen05.mma
// (kind::f16, fp16 operands, M=128, N=D, K=16) into one of two tensor-memory
// accumulators and commits to an mbarrier; while they run, the warps load and
// group the next tile's lookups and write the previous tile's pooled rows
// from the other accumulator (tcgen05.ld; the warp that reads lane quarter q
// gets the hi row of a bag in lane l and its lo row in lane l + 4).  After
// the MMAs, each warp clears the A entries it wrote (a list of their
// offsets, or its whole 8-row slab if the list overflowed).
//
// A uses the K-major layout with 128-byte swizzling: atoms of 8 rows x 64
// columns (1024 bytes), the 16-byte chunk c of row q of an atom stored at
// chunk c ^ q, so one bag's entries (one row, random columns) spread over all
// shared-memory banks; atoms are stacked 16 deep along M, then along K.
// W^T (written once per table) uses the no-swizzle K-major layout of
// 8x16-byte core matrices: element (n, k) at (n/8)*SBO + (k/8)*128 +
// (n%8)*16 + (k%8)*2.  Both take the table's rows padded to 64 as K.
//
// CTAs are persistent: each takes a contiguous range of (table, tile) items
// and loads a table's W^T when its range reaches it.  A tile whose outputs
// come out non-finite (inf or NaN inputs, or scales beyond every fp16 range)
// is pooled again by an fp32 gather.
#include "tbe_internal.cuh"
#include "tcgen05.cuh"

namespace tbe {

constexpr int kHistM = 128;          // MMA M: hi and lo rows of 64 bags
constexpr int kHistBags = 64;        // bags per tile
constexpr int kHistThreads = 512;    // 16 warps
constexpr int kHistWarps = kHistThreads / 32;
constexpr int kHistPre = 6;          // 32-lookup chunks of a warp held in registers ahead of the MMA wait
constexpr int kHistList = 256;       // A entries a warp remembers for its clear
constexpr uint32_t kNoKey = 0xffffffffu;

// Fallback for a tile whose tensor-core outputs are not finite: warp per
// bag, lanes over columns, fp32 accumulation straight from the table.
template <int DT, typename IDX>
__device__ void hist_tile_gather(const FwdArgs& a, const TableDesc& td, int t, int b0, int nb, int warp,
                                 int lane, bool& oob) {
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const int D = td.dim;
    for (int m = warp; m < nb; m += kHistWarps) {
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

// Power-of-two exponent e with x * 2^e in [2^14, 2^15) for a finite x > 0
// (from its exponent field: a normal x lies in [2^(E-127), 2^(E-126))),
// clamped to [-100, 100] so that 2^e and 2^-e are normal floats; 0 for zero,
// inf and NaN.
__device__ __forceinline__ int range_exp(float x) {
    const int E = (int)((__float_as_uint(x) >> 23) & 0xffu);
    if (!(x > 0.f) || E == 0xff) return 0;
    return tmax(-100, tmin(100, 141 - E));
}

// 2^e as a float, |e| <= 126.
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// Byte offset in A of row q (0..7) of 8-row group g, column k: the 128-byte
// swizzled K-major layout with 16 row groups (M = 128) per 64-column atom.
__device__ __forceinline__ uint32_t a_off(int g, int q, int k) {
    return (uint32_t)(k >> 6) * 16384u + (uint32_t)g * 1024u + (uint32_t)q * 128u +
           ((uint32_t)(((k >> 3) & 7) ^ q) << 4) + (uint32_t)(k & 7) * 2u;
}

// The table's W^T as fp16 (scaled by 2^f for bf16 tables) in the no-swizzle
// core-matrix layout: element (n, k) = W[k][n] * 2^f, zero for rows k >= R.
// All threads; returns f.
template <int DT>
__device__ int load_wt(const TableDesc& td, unsigned char* Ws, uint32_t sbo_b, int Kp, uint32_t* s_wmax) {
    const int tid = threadIdx.x;
    const int R = (int)td.rows, D = td.dim;
    const unsigned short* W = reinterpret_cast<const unsigned short*>(td.data);
    int f = 0;
    if constexpr (DT == DT_BF16) {
        if (tid == 0) *s_wmax = 0u;
        __syncthreads();
        uint32_t mx = 0u;  // bits of the largest finite magnitude (order of non-negative floats)
        for (int e = tid; e < R * (D / 8); e += kHistThreads) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(W) + e);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = fabsf(bf16_bits_to_float((w4[j >> 1] >> (16 * (j & 1))) & 0xffffu));
                if (isfinite(x)) mx = tmax(mx, __float_as_uint(x));
            }
        }
        atomicMax(s_wmax, mx);
        __syncthreads();
        f = range_exp(__uint_as_float(*s_wmax));
    }
    const float scale = pow2f(f);
    for (int e = tid; e < Kp * (D / 8); e += kHistThreads) {
        const int k = e / (D / 8), n8 = (e % (D / 8)) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k < R) v = __ldg(reinterpret_cast<const uint4*>(W + (int64_t)k * D + n8));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t bits = (w4[j >> 1] >> (16 * (j & 1))) & 0xffffu;
            if constexpr (DT == DT_BF16) bits = __half_as_ushort(__float2half_rn(bf16_bits_to_float(bits) * scale));
            *reinterpret_cast<unsigned short*>(Ws + core_off(n8 + j, k, sbo_b)) = (unsigned short)bits;
        }
    }
    return f;
}

// What the epilogue, the clear and the fallback need to know about a tile.
struct HistItem {
    int t, b0, nb, D, doff, kp;  // kp: the table's rows padded to 64
    float unscale;               // 2^-f of the table's W^T
};

template <int DT, typename IDX>
__global__ void __launch_bounds__(kHistThreads, 1)
    hist_kernel(FwdArgs a, const int32_t* hist_tables, int nhist, int dmax, uint32_t ab_bytes) {
    chain_wait();  // returns at once unless launched chained
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_wmax;
    __shared__ int s_nf[3];              // an epilogue saw non-finite outputs (indexed by iteration % 3)
    __shared__ int s_exp[3][kHistBags];  // e_b of the tiles in flight (indexed by item % 3)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (a.B + kHistBags - 1) / kHistBags;
    const int64_t total = (int64_t)nhist * ntiles;
    const int64_t it0 = total * blockIdx.x / gridDim.x;
    const int n = (int)(total * (blockIdx.x + 1) / gridDim.x - it0);
    if (n <= 0) return;  // whole CTA leaves before allocating anything
    // A (128 rows x kp, swizzle atoms 1024-byte aligned), then W^T (D x kp),
    // laid out for the table being processed; the warps' clear lists after
    // the largest such extent
    unsigned char* As = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t* s_list = reinterpret_cast<uint32_t*>(As + ab_bytes) + warp * kHistList;
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const uint32_t ncols = 2 * dmax <= 32 ? 32u : (2 * dmax <= 64 ? 64u : (2 * dmax <= 128 ? 128u : (2 * dmax <= 256 ? 256u : 512u)));
    const bool mean = a.mean != 0, weighted = a.weights != nullptr;
    bool oob = false, bad_off = false, timed_out = false;

    if (warp == 0) tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_nf[0] = s_nf[1] = s_nf[2] = 0;
    }
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = s_tmem;

    // lane l <= 4 of the warp: the offset starting the warp's bag l of an
    // item's tile (bags past B clamp to B); positions are clamped to
    // [-1, N + 1] (they are below 2^30)
    auto item_table = [&](int64_t item) { return __ldg(hist_tables + item / ntiles); };
    auto load_offs = [&](int64_t item) -> int32_t {
        const int t = item_table(item);
        const int b = tmin<int>((int)(item % ntiles) * kHistBags + 4 * warp + tmin(lane, 4), a.B);
        const int64_t v = ld_index(off, (int64_t)t * a.B + b);
        return (int32_t)tmin<int64_t>(tmax<int64_t>(v, -1), a.N + 1);
    };

    // Lanes holding one (bag, row) key form a group; the group's scales are
    // added in lane order and the lowest lane of the group (returns true)
    // keeps the sum.  Singletons skip the walk.
    auto group = [&](uint32_t key, bool valid, float s, float& acc) -> bool {
        const uint32_t grp = __match_any_sync(0xffffffffu, key);
        const uint32_t dup = __ballot_sync(0xffffffffu, valid && __popc(grp) > 1);
        acc = ((dup >> lane) & 1u) ? 0.f : s;
        for (uint32_t d = dup; d; d &= d - 1) {  // dup is the same in every lane
            const int src = __ffs(d) - 1;
            const float v = __shfl_sync(0xffffffffu, s, src);
            if ((grp >> src) & 1u) acc += v;
        }
        return valid && (__ffs(grp) - 1) == lane;
    };

    // Pooled rows of a finished tile whose tensor-core outputs were not
    // finite: again by an fp32 gather (all threads).
    auto fallback = [&](const HistItem& it) {
        hist_tile_gather<DT, IDX>(a, a.tabs[it.t], it.t, it.b0, it.nb, warp, lane, oob);
    };

    int32_t offv = load_offs(it0);
    int wt_table = -1;
    float wt_unscale = 1.f;
    uint32_t phase = 0;
    int lcnt = 0;  // entries in this warp's clear list (previous tile)
    HistItem prev{}, pp{}, epi{};

    for (int i = 0; i < n + 2; ++i) {
        const bool has_cur = i < n, has_prev = i >= 1 && i <= n, has_pp = i >= 2;
        if (tid == 0) s_nf[(i + 1) % 3] = 0;  // next iteration's flag (last read two iterations ago)
        HistItem cur{};
        TableDesc td{};
        // this warp's four bags: offsets and whether they rise monotonically
        int o0 = 0, o1 = 0, o2 = 0, o3 = 0, o4 = 0;
        bool all_valid = true;
        int prow[kHistPre];    // row of the lookup (-1: none, -2: out of range); after grouping, -1 unless group leader
        float pw[kHistPre];    // weight; after grouping, the group's scale sum
        if (has_cur) {
            const int64_t item = it0 + i;
            cur.t = item_table(item);
            td = a.tabs[cur.t];
            cur.b0 = (int)(item % ntiles) * kHistBags;
            cur.nb = tmin(kHistBags, a.B - cur.b0);
            cur.D = td.dim;
            cur.doff = td.doff;
            cur.kp = (int)((td.rows + 63) & ~int64_t(63));
            o0 = __shfl_sync(0xffffffffu, offv, 0);
            o1 = __shfl_sync(0xffffffffu, offv, 1);
            o2 = __shfl_sync(0xffffffffu, offv, 2);
            o3 = __shfl_sync(0xffffffffu, offv, 3);
            o4 = __shfl_sync(0xffffffffu, offv, 4);
            all_valid = o0 >= 0 && o0 <= o1 && o1 <= o2 && o2 <= o3 && o3 <= o4 && o4 <= a.N;
            if (i + 1 < n) offv = load_offs(it0 + i + 1);  // the next tile's, in flight from here
            // the first kHistPre chunks of the warp's lookups, in flight
            // across the epilogue below and the wait for the MMAs
#pragma unroll
            for (int c = 0; c < kHistPre; ++c) {
                const int p = o0 + 32 * c + lane;
                prow[c] = -1;
                pw[c] = 1.f;
                if (all_valid && p < o4) {
                    const int64_t x = ld_index(ind, p);
                    prow[c] = (x >= 0 && x < td.rows) ? (int)x : -2;
                    if (weighted) pw[c] = __ldg(a.weights + p);
                }
            }
        }

        // pooled rows of the tile before last (its MMAs finished one
        // iteration ago), from the accumulator it used
        if (has_pp) {
            epi = pp;
            const int q = warp & 3, l8 = lane & 7;
            const int u = 16 * q + 4 * (lane >> 3) + l8;  // bag within the tile (hi lanes)
            const bool st = l8 < 4 && u < pp.nb;
            const float s1 = st ? pow2f(-s_exp[(i - 2) % 3][u]) : 1.f;
            float* orow = a.out + (int64_t)(pp.b0 + u) * a.total_d + pp.doff;
            const uint32_t tcol = (uint32_t)(((i - 2) & 1) * dmax);
            bool nonfinite = false;
            for (int c = (warp >> 2) * 16; c < pp.D; c += (kHistWarps / 4) * 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + tcol + (uint32_t)c, v);  // whole warp
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float lo = __shfl_down_sync(0xffffffffu, v[k], 4);
                    v[k] = (v[k] + lo) * s1 * pp.unscale;
                }
                if (st) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) nonfinite |= !isfinite(v[k]);
                    if (a.vec_out) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            reinterpret_cast<float4*>(orow + c)[k] =
                                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) orow[c + k] = v[k];
                    }
                }
            }
            if (nonfinite) s_nf[i % 3] = 1;
        }

        // per bag: length, S_b = sum |s_i|, e_b; then the register chunks grouped
        float Lf0 = 0.f, Lf1 = 0.f, Lf2 = 0.f, Lf3 = 0.f;  // bag lengths
        float sc0 = 1.f, sc1 = 1.f, sc2 = 1.f, sc3 = 1.f;  // 2^e_b
        // scale of a lookup of bag j with weight w, times 2^e_j
        auto bag_scale = [&](int j, float w) {
            const float L = j == 0 ? Lf0 : j == 1 ? Lf1 : j == 2 ? Lf2 : Lf3;
            const float sc = j == 0 ? sc0 : j == 1 ? sc1 : j == 2 ? sc2 : sc3;
            return (mean ? __fdiv_rn(w, L) : w) * sc;
        };
        if (has_cur) {
            const int b = cur.b0 + 4 * warp;
            float S0, S1, S2, S3;
            {
                const int ob[5] = {o0, o1, o2, o3, o4};
                float Lf[4], S[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = b + j < a.B;
                    const bool ok = ob[j] >= 0 && ob[j] <= ob[j + 1] && ob[j + 1] <= a.N;
                    if (in && !ok) bad_off = true;
                    const int L = (in && ok) ? ob[j + 1] - ob[j] : 0;
                    Lf[j] = (float)L;
                    // unweighted: L ones (sum) or L copies of 1/L (mean)
                    S[j] = (mean && !weighted) ? (L > 0 ? 1.f : 0.f) : (float)L;
                }
                if (weighted) {
                    float part[4] = {0.f, 0.f, 0.f, 0.f};
                    if (all_valid) {
#pragma unroll
                        for (int c = 0; c < kHistPre; ++c) {
                            const int p = o0 + 32 * c + lane;
                            if (p < o4) {
                                const int j = (p >= o1) + (p >= o2) + (p >= o3);
                                const float s = fabsf(mean ? __fdiv_rn(pw[c], Lf[j]) : pw[c]);
#pragma unroll
                                for (int jj = 0; jj < 4; ++jj) part[jj] += jj == j ? s : 0.f;
                            }
                        }
                        for (int p = o0 + 32 * kHistPre + lane; p < o4; p += 32) {
                            const int j = (p >= o1) + (p >= o2) + (p >= o3);
                            const float w = __ldg(a.weights + p);
                            const float s = fabsf(mean ? __fdiv_rn(w, Lf[j]) : w);
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) part[jj] += jj == j ? s : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (Lf[j] > 0.f)
                                for (int p = ob[j] + lane; p < ob[j + 1]; p += 32) {
                                    const float w = __ldg(a.weights + p);
                                    part[j] += fabsf(mean ? __fdiv_rn(w, Lf[j]) : w);
                                }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) part[j] += __shfl_xor_sync(0xffffffffu, part[j], o);
                        S[j] = part[j];
                    }
                }
                Lf0 = Lf[0]; Lf1 = Lf[1]; Lf2 = Lf[2]; Lf3 = Lf[3];
                S0 = S[0]; S1 = S[1]; S2 = S[2]; S3 = S[3];
            }
            const int e0 = range_exp(S0), e1 = range_exp(S1), e2 = range_exp(S2), e3 = range_exp(S3);
            sc0 = pow2f(e0); sc1 = pow2f(e1); sc2 = pow2f(e2); sc3 = pow2f(e3);
            if (lane < 4) s_exp[i % 3][4 * warp + lane] = lane == 0 ? e0 : lane == 1 ? e1 : lane == 2 ? e2 : e3;
            // group the chunks held in registers
#pragma unroll
            for (int c = 0; c < kHistPre; ++c) {
                if (o0 + 32 * c >= o4) break;  // the warp's lookups end here (same in every lane)
                const int p = o0 + 32 * c + lane;
                const int j = (p >= o1) + (p >= o2) + (p >= o3);
                if (prow[c] == -2) oob = true;
                const bool valid = prow[c] >= 0;
                const uint32_t key = valid ? (((uint32_t)j << 16) | (uint32_t)prow[c]) : kNoKey;
                float acc;
                const bool lead = group(key, valid, bag_scale(j, pw[c]), acc);
                prow[c] = lead ? (int)key : -1;
                pw[c] = acc;
            }
        }

        // the previous tile's MMAs: wait; then redo the epilogue's tile by
        // gather if its outputs were not finite, and clear the A entries
        // the previous tile used
        if (has_prev) {
            const bool ok = mbar_wait(&s_bar, phase);
            if (__syncthreads_or(!ok)) {
                timed_out = true;
                break;
            }
            phase ^= 1u;
            tcgen05_after_sync();
            if (has_pp && s_nf[i % 3]) fallback(epi);
            if (lcnt <= kHistList) {
                for (int k = lane; k < lcnt; k += 32) {
                    const uint32_t e = s_list[k];
                    const int j = (int)(e >> 16), r = (int)(e & 0xffffu);
                    *reinterpret_cast<unsigned short*>(As + a_off(warp, j, r)) = 0;
                    *reinterpret_cast<unsigned short*>(As + a_off(warp, j + 4, r)) = 0;
                }
            } else {  // the warp's whole 8-row group, every 64-column atom
                for (int k = lane; k < prev.kp / 64 * 64; k += 32)
                    *reinterpret_cast<uint4*>(As + (uint32_t)(k >> 6) * 16384u + (uint32_t)warp * 1024u +
                                              (uint32_t)(k & 63) * 16u) = make_uint4(0u, 0u, 0u, 0u);
            }
            lcnt = 0;
            __syncwarp();
        }

        if (has_cur) {
            const int Kp = cur.kp;
            unsigned char* Ws = As + (size_t)kHistM * Kp * 2;
            const uint32_t sbo_b = (uint32_t)(Kp / 8) * 128u;
            if (cur.t != wt_table) {
                // a new table (the MMAs that read the old A and W^T have
                // finished): A laid out for its row count, all zero; its W^T
                for (int e = tid; e < kHistM * Kp * 2 / 16; e += kHistThreads)
                    reinterpret_cast<uint4*>(As)[e] = make_uint4(0u, 0u, 0u, 0u);
                wt_unscale = pow2f(-load_wt<DT>(td, Ws, sbo_b, Kp, &s_wmax));
                wt_table = cur.t;
                __syncthreads();  // A cleared before any warp writes its entries
            }
            cur.unscale = wt_unscale;
            // add one group sum into its entry (hi + lo) and remember the entry
            auto add_entry = [&](int key, float acc) {
                bool fresh = false;
                if (key >= 0) {
                    const int j = key >> 16, r = key & 0xffff;
                    unsigned short* ph = reinterpret_cast<unsigned short*>(As + a_off(warp, j, r));
                    unsigned short* pl = reinterpret_cast<unsigned short*>(As + a_off(warp, j + 4, r));
                    const float old = __half2float(__ushort_as_half(*ph)) + __half2float(__ushort_as_half(*pl));
                    const float x = old + acc;
                    const __half hi = __float2half_rn(x);
                    *ph = __half_as_ushort(hi);
                    *pl = __half_as_ushort(__float2half_rn(x - __half2float(hi)));
                    fresh = old == 0.f;
                }
                const uint32_t nf = __ballot_sync(0xffffffffu, fresh);
                if (fresh) {
                    const int slot = lcnt + __popc(nf & ((1u << lane) - 1u));
                    if (slot < kHistList) s_list[slot] = (uint32_t)key;
                }
                lcnt += __popc(nf);
                __syncwarp();  // the next chunk may read these entries
            };
            // one chunk of 32 positions from `base` (bag j fixed, or -1: by position)
            auto chunk = [&](int base, int end, int jfix) {
                const int p = base + lane;
                const int j = jfix >= 0 ? jfix : (p >= o1) + (p >= o2) + (p >= o3);
                int r = -1;
                float w = 1.f;
                if (p < end) {
                    const int64_t x = ld_index(ind, p);
                    if (x >= 0 && x < td.rows)
                        r = (int)x;
                    else
                        oob = true;
                    if (weighted) w = __ldg(a.weights + p);
                }
                const bool valid = r >= 0;
                const uint32_t key = valid ? (((uint32_t)j << 16) | (uint32_t)r) : kNoKey;
                float acc;
                const bool lead = group(key, valid, bag_scale(j, w), acc);
                add_entry(lead ? (int)key : -1, acc);
            };
            if (all_valid) {
#pragma unroll
                for (int c = 0; c < kHistPre; ++c) {
                    if (o0 + 32 * c >= o4) break;
                    add_entry(prow[c], pw[c]);
                }
                // chunks past the registers (warps whose bags hold more
                // than 32 * kHistPre lookups)
                for (int base = o0 + 32 * kHistPre; base < o4; base += 32) chunk(base, o4, -1);
            } else {
                // offsets that do not rise monotonically: each valid bag on its own
                const int ob[5] = {o0, o1, o2, o3, o4};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float L = j == 0 ? Lf0 : j == 1 ? Lf1 : j == 2 ? Lf2 : Lf3;
                    if (!(L > 0.f)) continue;
                    for (int base = ob[j]; base < ob[j + 1]; base += 32) chunk(base, ob[j + 1], j);
                }
            }
            fence_proxy_async_smem();  // generic-proxy writes of A and W^T -> tensor cores
            tcgen05_before_sync();
            __syncthreads();
            tcgen05_after_sync();
            if (tid == 0) {
                const uint32_t idesc = mma_idesc(0, kHistM, cur.D);  // fp16 x fp16 -> fp32
                const uint64_t adesc = smem_desc_sw128(smem_u32(As), 1024u);
                const uint64_t bdesc = smem_desc(smem_u32(Ws), 128u, sbo_b);
                const uint32_t d = tmem + (uint32_t)((i & 1) * dmax);
                // K step j (16 columns): A's start moves 32 bytes within a
                // 64-column atom and 16 KB per atom; W^T's by 256 bytes (the
                // address field, address >> 4, does not carry: addresses < 2^18)
                for (int j = 0; j < Kp / 16; ++j)
                    mma_f16(d, adesc + (uint64_t)((j >> 2) * 1024 + (j & 3) * 2), bdesc + (uint64_t)(16 * j), idesc,
                            j > 0 ? 1u : 0u);
                mma_commit(&s_bar);
            }
        }
        pp = prev;
        prev = cur;
    }
    if (timed_out) {
        if (tid == 0) atomicOr(&a.blk->error, ERR_TIMEOUT);
        mbar_wait(&s_bar, phase);  // a second bounded wait for the MMAs in flight
    } else {
        __syncthreads();  // the last epilogue (no wait followed it)
        if (s_nf[(n + 1) % 3]) fallback(epi);
    }
    if (oob) atomicOr(&a.blk->error, ERR_OOB);
    if (bad_off) atomicOr(&a.blk->error, ERR_OFFSETS);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

// Bytes of A and W^T for a table of `rows` rows and dim D (K: rows padded to 64).
size_t hist_ab_bytes(int64_t rows, int dim) { return (size_t)(kHistM + dim) * (size_t)((rows + 63) & ~int64_t(63)) * 2; }

// Dynamic shared memory of a histogram launch: room to align A to 1024
// bytes, the largest A + W^T extent of its tables, the warps' clear lists.
size_t hist_smem_bytes(size_t ab_bytes) { return 1024 + ab_bytes + sizeof(uint32_t) * kHistWarps * kHistList; }

// The launches' dynamic shared-memory limit, raised to the device's opt-in
// maximum less the kernel's static shared memory (on the current device; the
// attribute is per device).
cudaError_t hist_configure(int optin) {
    const void* fns[4] = {(const void*)hist_kernel<DT_F16, int32_t>, (const void*)hist_kernel<DT_F16, int64_t>,
                          (const void*)hist_kernel<DT_BF16, int32_t>, (const void*)hist_kernel<DT_BF16, int64_t>};
    for (const void* f : fns) {
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, f);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int DT, typename IDX>
static cudaError_t launch_hist_t(const FwdArgs& a, const HistGroup& g, cudaStream_t s) {
    const int ntiles = (a.B + kHistBags - 1) / kHistBags;
    const int64_t items = (int64_t)g.n * ntiles;
    const int sms = a.num_sms > 0 ? a.num_sms : 1;
    const unsigned grid = (unsigned)tmin<int64_t>(items, sms);
    // the forward's long-bag kernel (or the other dtype's launch) runs just before
    return launch_chained_smem(hist_kernel<DT, IDX>, dim3(grid), dim3(kHistThreads), g.smem, s, a, g.tables, g.n,
                               g.dmax, (uint32_t)g.ab_bytes);
}

// One launch per table dtype (f16, bf16) that has histogram tables.
cudaError_t launch_hist(const FwdArgs& a, const HistGroup& f16, const HistGroup& bf16, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (f16.n > 0)
        e = a.idx64 ? launch_hist_t<DT_F16, int64_t>(a, f16, s) : launch_hist_t<DT_F16, int32_t>(a, f16, s);
    if (e == cudaSuccess && bf16.n > 0)
        e = a.idx64 ? launch_hist_t<DT_BF16, int64_t>(a, bf16, s) : launch_hist_t<DT_BF16, int32_t>(a, bf16, s);
    return e;
}

}  // namespace tbe
