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
// are multiplied by a power of two 2^e_b chosen from M_b = L_b * max |s_i|
// (every |H[b, r]| <= M_b): M_b * 2^e_b lies in [2^14, 2^15), far from fp16's
// overflow, and an entry loses relative precision only where it is below
// M_b * 2^-28.  fp16 tables enter as they are; a bf16 table is multiplied by
// a power of two 2^f chosen from its largest magnitude the same way, which is
// exact for every value within 2^29 of that magnitude.  The products and sums
// are fp32 in tensor memory; the epilogue adds the hi and lo products and
// multiplies by 2^-e_b and 2^-f.
//
// Schedule.  A tile is 64 bags.  The MMA's A operand (M = 128 rows) holds hi
// and lo of the tile's 64 bags; the 8-row group g of A belongs to builder
// warp g: its rows 0-3 are hi of the warp's four bags, rows 4-7 their lo.
// Each builder warp walks its four bags' lookups (contiguous positions) 32 at
// a time; lanes with the same (bag, row) are grouped with a warp match, the
// group's scales are added in lane order, and one lane adds the group sum
// into the H entry (read hi + lo, add, split again).  A warp owns its rows of
// A, so no two warps touch one entry: no atomics, and the result does not
// depend on scheduling.
//
// The warps never wait for one another at a CTA barrier.  A warp that has
// written its rows of a tile (and its share of a new table's W^T) counts
// itself in with an acquire-release atomic; the last of the 16 issues the
// tile's Kp/16 tcgen05.mma (kind::f16, fp16 operands, M=128, N=D, K=16) into
// one of two tensor-memory accumulators and commits them to the mbarrier
// "done" (which it also arrives on, so what the warps published reaches
// whoever waits on "done").  A warp waits on "done" of the previous tile
// before it clears and rewrites its rows; until
// then it loads and groups the next tile's lookups and writes the pooled
// rows of the tile before from the other accumulator (tcgen05.ld: the warp
// that reads lane quarter q gets the hi row of a bag in lane l and its lo
// row in lane l + 4).  A lane whose pooled values come out non-finite (inf or
// NaN inputs, or scales beyond every fp16 range) pools its bag's columns
// again by an fp32 gather.
//
// A uses the K-major layout with 128-byte swizzling: atoms of 8 rows x 64
// columns (1024 bytes), the 16-byte chunk c of row q of an atom stored at
// chunk c ^ q, so one bag's entries (one row, random columns) spread over all
// shared-memory banks; atoms are stacked 16 deep along M, then along K, for
// the largest row count of the launch's tables.  W^T uses the no-swizzle
// K-major layout of 8x16-byte core matrices: element (n, k) at
// (n/8)*SBO + (k/8)*128 + (n%8)*16 + (k%8)*2.  Both take the table's rows
// padded to 64 as K.
//
// CTAs are persistent: each takes a contiguous range of (table, tile) items
// and loads a table's W^T when its range reaches it.
#include "tbe_internal.cuh"
#include "tcgen05.cuh"

namespace tbe {

constexpr int kHistM = 128;          // MMA M: hi and lo rows of 64 bags
constexpr int kHistBags = 64;        // bags per tile
constexpr int kHistWarps = 16;       // warps, four bags each
constexpr int kHistThreads = 32 * kHistWarps;
constexpr int kHistPre = 6;          // 32-lookup chunks of a warp held in registers ahead of the wait
constexpr int kHistList = 256;       // A entries a warp remembers for its clear
constexpr uint32_t kNoKey = 0xffffffffu;

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

// The lo term of an entry (row q + 4) sits 512 bytes after its hi term (row
// q), with its 16-byte chunk index XOR 4 (q + 4 = q ^ 4 for q < 4): 512 + 64
// or 512 - 64 bytes further.
__device__ __forceinline__ uint32_t lo_off(uint32_t hi) { return hi + 512u + ((hi & 64u) ? 0u - 64u : 64u); }

// What the epilogue and the clear need to know about a tile.
struct HistItem {
    int t, b0, nb, D, doff;
    float unscale;  // 2^-f of the table's W^T
};

// One lane: bag b of table t, columns [c, c + 16), by an fp32 gather
// straight from the table (the fallback for non-finite tensor-core results).
template <int DT, typename IDX>
__device__ void lane_gather(const FwdArgs& a, const TableDesc& td, int t, int b, int c, float (&v)[16],
                            bool& oob) {
    const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
    const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
    const int64_t bag = (int64_t)t * a.B + b;
    int64_t start = ld_index(off, bag), end = ld_index(off, bag + 1);
    if (start < 0 || end < start || end > a.N) start = end = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = 0.f;
    for (int64_t p = start; p < end; ++p) {
        const int64_t x = ld_index(ind, p);
        if (x < 0 || x >= td.rows) {
            oob = true;
            continue;
        }
        const float s = a.weights ? __ldg(a.weights + p) : 1.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = fmaf(s, load_elem<DT>(td.data, x * td.dim + c + k), v[k]);
    }
    if (a.mean && end > start)
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = __fdiv_rn(v[k], (float)(end - start));
}

// This warp's share (rows k = warp, warp + 16, ...) of the table's W^T as
// fp16, scaled by 2^f for bf16 tables, in the no-swizzle core-matrix layout:
// element (n, k) = W[k][n] * 2^f, zero for rows k >= R.  Returns f (each warp
// finds the same: a bf16 table's largest magnitude is read by every warp).
template <int DT>
__device__ int load_wt_part(const TableDesc& td, unsigned char* Ws, int kp, int warp, int lane) {
    const int R = (int)td.rows, D = td.dim;
    const uint32_t sbo = (uint32_t)(kp / 8) * 128u;
    const unsigned short* W = reinterpret_cast<const unsigned short*>(td.data);
    int f = 0;
    if constexpr (DT == DT_BF16) {
        uint32_t mx = 0u;  // bits of the largest finite magnitude (order of non-negative floats)
        for (int e = lane; e < R * (D / 8); e += 32) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(W) + e);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = fabsf(bf16_bits_to_float((w4[j >> 1] >> (16 * (j & 1))) & 0xffffu));
                if (isfinite(x)) mx = tmax(mx, __float_as_uint(x));
            }
        }
        f = range_exp(__uint_as_float(__reduce_max_sync(0xffffffffu, mx)));
    }
    const float scale = pow2f(f);
    const int nv = D / 8;  // 16-byte vectors per row
    for (int e = lane; e < (kp / kHistWarps) * nv; e += 32) {
        const int k = warp + kHistWarps * (e / nv), n8 = (e % nv) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k < R) v = __ldg(reinterpret_cast<const uint4*>(W + (int64_t)k * D + n8));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t bits = (w4[j >> 1] >> (16 * (j & 1))) & 0xffffu;
            if constexpr (DT == DT_BF16) bits = __half_as_ushort(__float2half_rn(bf16_bits_to_float(bits) * scale));
            *reinterpret_cast<unsigned short*>(Ws + core_off(n8 + j, k, sbo)) = (unsigned short)bits;
        }
    }
    return f;
}

template <int DT, typename IDX>
__global__ void __launch_bounds__(kHistThreads, 1)
    hist_kernel(FwdArgs a, const int32_t* hist_tables, int nhist, int dmax, int kmax, uint32_t wt_bytes) {
    chain_wait();  // returns at once unless launched chained
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint32_t s_count[2];      // warps done writing a tile (indexed by item % 2)
    __shared__ uint64_t s_done;          // a tile's MMAs finished (commit) + issued (the issuing thread): 2 arrivals
    __shared__ uint32_t s_tmem;
    __shared__ int s_issued;             // tiles whose MMAs were issued
    __shared__ int s_exp[3][kHistBags];  // e_b of the tiles in flight (indexed by item % 3)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (a.B + kHistBags - 1) / kHistBags;
    const int64_t total = (int64_t)nhist * ntiles;
    const int64_t it0 = total * blockIdx.x / gridDim.x;
    const int n = (int)(total * (blockIdx.x + 1) / gridDim.x - it0);
    if (n <= 0) return;  // whole CTA leaves before allocating anything
    // A (128 rows x kmax; swizzle atoms 1024-byte aligned), W^T (D x kp of
    // the table being processed), the builder warps' clear lists
    unsigned char* As = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* Ws = As + (size_t)kHistM * kmax * 2;
    const uint32_t ncols = 2 * dmax <= 32 ? 32u : (2 * dmax <= 64 ? 64u : (2 * dmax <= 128 ? 128u : (2 * dmax <= 256 ? 256u : 512u)));
    bool oob = false, bad_off = false, timed_out = false;

    if (warp == 0) tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        mbar_init(&s_done, 2);
        s_count[0] = s_count[1] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_issued = 0;
    }
    for (int e = tid; e < kHistM * kmax * 2 / 16; e += kHistThreads)
        reinterpret_cast<uint4*>(As)[e] = make_uint4(0u, 0u, 0u, 0u);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = s_tmem;

    {
        const IDX* off = reinterpret_cast<const IDX*>(a.offsets);
        const IDX* ind = reinterpret_cast<const IDX*>(a.indices);
        uint32_t* s_list = reinterpret_cast<uint32_t*>(Ws + wt_bytes) + warp * kHistList;
        const bool mean = a.mean != 0, weighted = a.weights != nullptr;

        // lane l <= 4: the offset starting the warp's bag l of an item's tile
        // (bags past B clamp to B); positions clamped to [-1, N + 1] (they
        // are below 2^30)
        // items walk (table k, tile) in order: the next item's position is
        // kept incrementally (no divisions per tile)
        int nk = (int)(it0 / ntiles), ntile = (int)(it0 - (int64_t)nk * ntiles);  // next item to load
        int ck = nk, ctile = ntile;                                                // current item
        auto load_offs = [&](int k, int tile) -> int32_t {
            const int t = __ldg(hist_tables + k);
            const int b = tmin<int>(tile * kHistBags + 4 * warp + tmin(lane, 4), a.B);
            const int64_t v = ld_index(off, (int64_t)t * a.B + b);
            return (int32_t)tmin<int64_t>(tmax<int64_t>(v, -1), a.N + 1);
        };
        auto advance = [&](int& k, int& tile) {
            if (++tile == ntiles) {
                tile = 0;
                ++k;
            }
        };

        // Lanes holding one (bag, row) key form a group; the group's scales
        // are added in lane order and the lowest lane of the group (returns
        // true) keeps the sum.  Singletons skip the walk.
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

        int32_t offv = load_offs(nk, ntile);
        advance(nk, ntile);
        int wt_table = -1;
        float wt_unscale = 1.f;
        int lcnt = 0;  // entries in this warp's clear list (previous tile)
        HistItem prev{}, pp{};

        for (int i = 0; i < n + 2; ++i) {
            const bool has_cur = i < n, has_prev = i >= 1 && i <= n, has_pp = i >= 2;
            HistItem cur{};
            TableDesc td{};
            // this warp's four bags: offsets, and whether they rise monotonically
            int o0 = 0, o1 = 0, o2 = 0, o3 = 0, o4 = 0;
            bool all_valid = true;
            int prow[kHistPre];  // row of the lookup (-1: none, -2: out of range); after grouping: key of a group leader, else -1
            float pw[kHistPre];  // weight; after grouping: the group's scale sum
            if (has_cur) {
                cur.t = __ldg(hist_tables + ck);
                td = a.tabs[cur.t];
                cur.b0 = ctile * kHistBags;
                advance(ck, ctile);
                cur.nb = tmin(kHistBags, a.B - cur.b0);
                cur.D = td.dim;
                cur.doff = td.doff;
                o0 = __shfl_sync(0xffffffffu, offv, 0);
                o1 = __shfl_sync(0xffffffffu, offv, 1);
                o2 = __shfl_sync(0xffffffffu, offv, 2);
                o3 = __shfl_sync(0xffffffffu, offv, 3);
                o4 = __shfl_sync(0xffffffffu, offv, 4);
                all_valid = o0 >= 0 && o0 <= o1 && o1 <= o2 && o2 <= o3 && o3 <= o4 && o4 <= a.N;
                if (i + 1 < n) {  // the next tile's, in flight from here
                    offv = load_offs(nk, ntile);
                    advance(nk, ntile);
                }
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

            // pooled rows of the tile before last (its MMAs finished before
            // the previous iteration's wait returned), from its accumulator
            if (has_pp) {
                const int q = warp & 3, l8 = lane & 7;
                const int u = 16 * q + 4 * (lane >> 3) + l8;  // bag within the tile (hi lanes)
                const bool st = l8 < 4 && u < pp.nb;
                const float s1 = st ? pow2f(-s_exp[(i - 2) % 3][u]) : 1.f;
                float* orow = a.out + (int64_t)(pp.b0 + u) * a.total_d + pp.doff;
                const uint32_t tcol = (uint32_t)(((i - 2) & 1) * dmax);
                for (int c = (warp >> 2) * 16; c < pp.D; c += (kHistWarps / 4) * 16) {
                    float v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + tcol + (uint32_t)c, v);  // whole warp
                    float chk = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float lo = __shfl_down_sync(0xffffffffu, v[k], 4);
                        v[k] = (v[k] + lo) * s1 * pp.unscale;
                        chk += v[k] * 0.f;  // NaN if any value is inf or NaN
                    }
                    if (st) {
                        if (chk != 0.f || !isfinite(chk)) {
                            // recomputed by fp32 gather (inf and NaN where the definition puts them)
                            lane_gather<DT, IDX>(a, a.tabs[pp.t], pp.t, pp.b0 + u, c, v, oob);
                        }
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
            }

            // per bag: length, M_b = L_b * max |s_i|, e_b; the register chunks grouped
            float Lf0 = 0.f, Lf1 = 0.f, Lf2 = 0.f, Lf3 = 0.f;  // bag lengths
            float sc0 = 1.f, sc1 = 1.f, sc2 = 1.f, sc3 = 1.f;  // 2^e_b
            int e0 = 0, e1 = 0, e2 = 0, e3 = 0;
            // scale of a lookup of bag j with weight w, times 2^e_j
            auto bag_scale = [&](int j, float w) {
                const float L = j == 0 ? Lf0 : j == 1 ? Lf1 : j == 2 ? Lf2 : Lf3;
                const float sc = j == 0 ? sc0 : j == 1 ? sc1 : j == 2 ? sc2 : sc3;
                return (mean ? __fdiv_rn(w, L) : w) * sc;
            };
            if (has_cur) {
                const int b = cur.b0 + 4 * warp;
                const int ob[5] = {o0, o1, o2, o3, o4};
                float Lf[4], M[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = b + j < a.B;
                    const bool ok = ob[j] >= 0 && ob[j] <= ob[j + 1] && ob[j + 1] <= a.N;
                    if (in && !ok) bad_off = true;
                    const int L = (in && ok) ? ob[j + 1] - ob[j] : 0;
                    Lf[j] = (float)L;
                    M[j] = (mean && !weighted) ? (L > 0 ? 1.f : 0.f) : (float)L;  // unweighted: L * 1 or L * 1/L
                }
                if (weighted) {
                    // the largest |w| of each bag (the bits of non-negative
                    // floats order like the floats)
                    uint32_t mx[4] = {0u, 0u, 0u, 0u};
                    if (all_valid) {
#pragma unroll
                        for (int c = 0; c < kHistPre; ++c) {
                            const int p = o0 + 32 * c + lane;
                            const int j = (p >= o1) + (p >= o2) + (p >= o3);
                            const uint32_t wb = p < o4 ? __float_as_uint(fabsf(pw[c])) : 0u;
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) mx[jj] = tmax(mx[jj], jj == j ? wb : 0u);
                        }
                        for (int p = o0 + 32 * kHistPre + lane; p < o4; p += 32) {
                            const int j = (p >= o1) + (p >= o2) + (p >= o3);
                            const uint32_t wb = __float_as_uint(fabsf(__ldg(a.weights + p)));
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) mx[jj] = tmax(mx[jj], jj == j ? wb : 0u);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (Lf[j] > 0.f)
                                for (int p = ob[j] + lane; p < ob[j + 1]; p += 32)
                                    mx[j] = tmax(mx[j], __float_as_uint(fabsf(__ldg(a.weights + p))));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float wmax = __uint_as_float(__reduce_max_sync(0xffffffffu, mx[j]));
                        // a NaN weight makes every value unbounded: e = 0 and the
                        // tile's non-finite outputs take the gather
                        M[j] = isnan(wmax) ? 0.f : Lf[j] * (mean ? wmax / fmaxf(Lf[j], 1.f) : wmax);
                    }
                }
                e0 = range_exp(M[0]); e1 = range_exp(M[1]); e2 = range_exp(M[2]); e3 = range_exp(M[3]);
                sc0 = pow2f(e0); sc1 = pow2f(e1); sc2 = pow2f(e2); sc3 = pow2f(e3);
                Lf0 = Lf[0]; Lf1 = Lf[1]; Lf2 = Lf[2]; Lf3 = Lf[3];
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

            // the previous tile's MMAs: wait, then clear the A entries it used
            if (has_prev) {
                if (!mbar_wait(&s_done, (uint32_t)((i - 1) & 1))) {
                    timed_out = true;
                    break;
                }
                tcgen05_after_sync();
                if (lcnt <= kHistList) {
                    for (int k = lane; k < lcnt; k += 32) {
                        const uint32_t e = s_list[k];
                        const int j = (int)(e >> 16), r = (int)(e & 0xffffu);
                        const uint32_t o = a_off(warp, j, r);
                        *reinterpret_cast<unsigned short*>(As + o) = 0;
                        *reinterpret_cast<unsigned short*>(As + lo_off(o)) = 0;
                    }
                } else {  // the warp's whole 8-row group, every 64-column atom
                    for (int k = lane; k < kmax; k += 32)
                        *reinterpret_cast<uint4*>(As + (uint32_t)(k >> 6) * 16384u + (uint32_t)warp * 1024u +
                                                  (uint32_t)(k & 63) * 16u) = make_uint4(0u, 0u, 0u, 0u);
                }
                lcnt = 0;
                __syncwarp();
            }

            if (has_cur) {
                if (cur.t != wt_table) {  // a new table; the MMAs that read the old W^T have finished
                    wt_unscale = pow2f(-load_wt_part<DT>(td, Ws, (int)((td.rows + 63) & ~int64_t(63)), warp, lane));
                    wt_table = cur.t;
                }
                cur.unscale = wt_unscale;
                if (lane < 4) s_exp[i % 3][4 * warp + lane] = lane == 0 ? e0 : lane == 1 ? e1 : lane == 2 ? e2 : e3;
                // add one group sum into its entry (hi + lo) and remember the entry
                auto add_entry = [&](int key, float acc) {
                    bool fresh = false;
                    if (key >= 0) {
                        const int j = key >> 16, r = key & 0xffff;
                        const uint32_t o = a_off(warp, j, r);
                        unsigned short* ph = reinterpret_cast<unsigned short*>(As + o);
                        unsigned short* pl = reinterpret_cast<unsigned short*>(As + lo_off(o));
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
                // publish the A rows (and W^T) to the tensor cores and this
                // warp's writes and tensor-memory reads (the epilogue above)
                // to the warp that issues the MMAs: the last one to count in
                fence_proxy_async_smem();
                tcgen05_before_sync();
                __syncwarp();
                if (lane == 0) {
                    uint32_t before;
                    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                                 : "=r"(before)
                                 : "r"(smem_u32(&s_count[i & 1]))
                                 : "memory");
                    if (before == kHistWarps - 1) {
                        // every warp's part of the tile is in; the count is
                        // reused two tiles on, after everyone has waited on
                        // this tile's "done"
                        *reinterpret_cast<volatile uint32_t*>(&s_count[i & 1]) = 0u;
                        tcgen05_after_sync();
                        const int kp = (int)((td.rows + 63) & ~int64_t(63));
                        const uint32_t idesc = mma_idesc(0, kHistM, cur.D);  // fp16 x fp16 -> fp32
                        const uint64_t adesc = smem_desc_sw128(smem_u32(As), 1024u);
                        const uint64_t bdesc = smem_desc(smem_u32(Ws), 128u, (uint32_t)(kp / 8) * 128u);
                        const uint32_t d = tmem + (uint32_t)((i & 1) * dmax);
                        // K step j (16 columns): A's start moves 32 bytes within a
                        // 64-column atom and 16 KB per atom; W^T's by 256 bytes (the
                        // address field, address >> 4, does not carry: addresses < 2^18)
                        for (int j = 0; j < kp / 16; ++j)
                            mma_f16(d, adesc + (uint64_t)((j >> 2) * 1024 + (j & 3) * 2), bdesc + (uint64_t)(16 * j),
                                    idesc, j > 0 ? 1u : 0u);
                        mma_commit(&s_done);
                        mbar_arrive(&s_done);
                        s_issued = i + 1;
                    }
                }
                __syncwarp();
            }
            pp = prev;
            prev = cur;
        }
    }
    if (__syncthreads_or(timed_out)) {
        if (tid == 0) {
            atomicOr(&a.blk->error, ERR_TIMEOUT);
            if (s_issued > 0) mbar_wait(&s_done, (uint32_t)((s_issued - 1) & 1));  // the MMAs in flight (bounded)
        }
    }
    if (oob) atomicOr(&a.blk->error, ERR_OOB);
    if (bad_off) atomicOr(&a.blk->error, ERR_OFFSETS);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

// Dynamic shared memory of a histogram launch whose tables have at most
// kmax rows (padded to 64) and at most wt_bytes of W^T: room to align A to
// 1024 bytes, A (128 rows x kmax fp16), W^T, the builder warps' clear lists.
size_t hist_smem_bytes(int kmax, size_t wt_bytes) {
    return 1024 + (size_t)kHistM * kmax * 2 + wt_bytes + sizeof(uint32_t) * kHistWarps * kHistList;
}

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
                               g.dmax, g.kmax, (uint32_t)g.wt_bytes);
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
