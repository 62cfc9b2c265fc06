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
//    consecutive bag ranges) and walks its bags 32 at a time.  Per tile:
//     - every thread takes lookups of the tile by position, finds its bag
//       (a shuffle search over the tile's bag offsets) and adds its scale to
//       an fp32 histogram in shared memory (shared-memory atomics; a bag's
//       lookups are spread over the CTA's threads);
//     - the touched histogram entries are split into three bf16 terms
//       x = x0 + x1 + x2 (24 significant bits) and written into H^T (rows x
//       bags, no-swizzle K-major core matrices); G_t (columns x bags) is
//       split the same way;
//     - one thread issues tcgen05.mma (kind::f16, bf16 operands, fp32
//       accumulator in tensor memory, M = 128, N = dim, K = 16) for the six
//       products x_i y_j with i + j <= 2, and commits to an mbarrier.
//    The lookup that finds a histogram entry empty owns it: it writes the
//    entry's H^T terms and clears the entry for the next tile.  While the
//    tensor cores run, the threads build the next tile's histogram and G_t
//    (G_t is double-buffered); after the MMAs, the owners clear their H^T
//    entries.  Every kDensePromote tiles the tensor-memory accumulator is
//    added (fp32, round to nearest) into a second tensor-memory sum and
//    restarted, so the tensor cores' own accumulation rounds against a small
//    partial sum.  At the end the CTA stores that sum into its own slice of
//    the gradient buffer and marks the rows its lookups touched.
//  dense_update_kernel: one warp per row of every dense table; a row that
//    some lookup touched adds its S partial sums in order, gets its optimizer
//    step (the same SGD / row-wise Adagrad arithmetic as the sorted path) and
//    is stored once.
//
// Repeated lookups of one row in one bag meet in a shared-memory fp32
// atomic; their order (and so the last bit of such an entry when the scales
// are not integers) may vary from run to run.
#include "tbe_internal.cuh"
#include "tcgen05.cuh"

namespace tbe {

constexpr int kDenseThreads = 512;
constexpr int kDenseWarps = kDenseThreads / 32;
constexpr int kMmaWarp = kDenseWarps - 1;              // issues the MMAs and takes no lookups
constexpr int kDenseWorkers = kDenseThreads - 32;      // threads of the other warps
constexpr int kDenseKT = 32;      // bags per tile (two MMA K steps)
constexpr int kDenseSplit = 3;    // bf16 terms per operand
constexpr int kDenseLk = 5;       // lookups per worker thread per tile remembered for the sparse clears
constexpr int kDensePromote = 4;  // tiles summed in the tensor-memory accumulator before it is restarted
constexpr uint32_t kNoEntry = 0xffffffffu;
constexpr int kDenseTab = kDenseWorkers * kDenseLk;  // lookups of a tile whose bag is tabulated

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

// Shared-memory plan of one CTA for Mp rows and dim D (bytes): H^T terms,
// two buffers of G_t terms, the fp32 histogram, the touched-row flags.
__host__ __device__ inline size_t dense_a_bytes(int Mp) { return (size_t)Mp * kDenseKT * 2; }
__host__ __device__ inline size_t dense_b_bytes(int D) { return (size_t)D * kDenseKT * 2; }
__host__ __device__ inline size_t dense_smem_bytes(int Mp, int D) {
    return kDenseSplit * dense_a_bytes(Mp) + 2 * kDenseSplit * dense_b_bytes(D) +
           sizeof(float) * (size_t)Mp * kDenseKT + sizeof(uint32_t) * (size_t)Mp;
}

__host__ __device__ inline uint32_t dense_tmem_cols(int n) {
    return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

// Histogram entry (m, j): row-major [Mp][32] with the bag index swizzled by
// the row, so the lanes of a warp (mostly one bag, many rows) hit different
// banks.
__device__ __forceinline__ uint32_t hf_index(uint32_t m, uint32_t j) { return m * kDenseKT + (j ^ (m & 31u)); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__global__ void __launch_bounds__(kDenseThreads, 1) dense_mma_kernel(DenseArgs a, Workspace ws, int groups_max) {
    extern __shared__ __align__(1024) unsigned char dsm[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    __shared__ uint8_t s_bagtab[2][kDenseTab];  // bag of each lookup, for two tiles
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
    unsigned char* Bs = dsm + kDenseSplit * dense_a_bytes(Mp);  // [buffer][split][D x KT] bf16
    float* Hf = reinterpret_cast<float*>(Bs + 2 * kDenseSplit * dense_b_bytes(D));  // [Mp][KT] fp32
    uint32_t* s_cnt = reinterpret_cast<uint32_t*>(Hf + (size_t)Mp * kDenseKT);     // [Mp]
    const uint32_t sbo = (uint32_t)(kDenseKT / 8) * 128u;  // bytes per 8 rows (K-major core matrices)

    // bag range of this part
    const int bk0 = (int)(((int64_t)a.B * sp) / splits);
    const int bk1 = (int)(((int64_t)a.B * (sp + 1)) / splits);
    const int ntiles = (bk1 - bk0 + kDenseKT - 1) / kDenseKT;
    const uint32_t* boff = ws.dboff + (int64_t)td.dslot * (a.B + 1);
    const bool has_scale = ws.counters[CTR_HAS_SCALE] != 0;
    const uint32_t ncols = dense_tmem_cols(2 * mtiles * D);  // short and long accumulators
    const uint32_t long0 = (uint32_t)(mtiles * D);           // first column of the long one
    if (warp == 0) tmem_alloc(&s_tmem, ncols);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {
        uint4* pa = reinterpret_cast<uint4*>(As);
        const int n16 = (int)(kDenseSplit * dense_a_bytes(Mp) / 16);
        for (int i = tid; i < n16; i += kDenseThreads) pa[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < Mp * kDenseKT; i += kDenseThreads) Hf[i] = 0.f;
        for (int i = tid; i < Mp; i += kDenseThreads) s_cnt[i] = 0;
    }
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = mma_idesc(1, 128, D);  // bf16 x bf16 -> fp32
    const uint32_t abase = smem_u32(As), bbase = smem_u32(Bs);
    // Descriptors of the tile's operands, computed in registers when the MMAs
    // are issued: the start address field (bits 0-13, address >> 4) of the
    // base descriptors plus the byte offset of the split term, the M tile and
    // the K step >> 4 (addresses stay below 2^18 bytes, so the field does
    // not carry).
    const uint64_t adesc0 = smem_desc(abase, 128u, sbo);
    const uint64_t bdesc0 = smem_desc(bbase, 128u, sbo);
    const uint32_t a_split16 = (uint32_t)(dense_a_bytes(Mp) >> 4), b_split16 = (uint32_t)(dense_b_bytes(D) >> 4);
    const uint32_t mtile16 = (16u * sbo) >> 4, kstep16 = 256u >> 4;
    __syncthreads();

    // A tile's inputs, loaded into registers one tile ahead so their latency
    // hides behind the previous tile's work: the bag offsets (lane l: first
    // lookup of bag l), the row and scale of this thread's lookups
    // q0 + perm + 480*kk, and the gradient values of its G_t items (a warp
    // item covers 8 columns x 8 bags; lane: column c0 + lane%8, bags
    // 2*(lane/8) and +1, so each split term is one 4-byte store and a warp's
    // stores fill distinct banks).
    constexpr int kGItems = 4;  // G_t items per warp held in registers (dim <= 128; dim 256 loads the rest in place)
    struct TileIn {
        int b0, nb;
        uint32_t q0, qend, ol;
        int r[kDenseLk];
        float s[kDenseLk];
        float g[2 * kGItems];
    };
    // lookup slot of worker thread t in every block of 480 positions:
    // (t % 8) * 60 + t / 8, so a warp's 32 lookups come from 8 runs of 4
    // (mostly 8 bags: their H^T entries spread over the shared-memory banks);
    // the MMA warp takes no lookups, so issuing the MMAs (which can wait for
    // room in the tensor pipe) delays no histogram work
    const bool worker = warp < kMmaWarp;
    const int perm = (tid & 7) * (kDenseWorkers / 8) + (tid >> 3);
    const int bitems = (D / 8) * (kDenseKT / 8);
    // item it covers columns 8*(it % (D/8)) .. +7 and bags 8*(it / (D/8)) .. +7;
    // this lane's column and first bag for item `it`
    auto item_cj = [&](int it, int& c, int& j) {
        const int cg = it % (D / 8);
        c = cg * 8 + (lane & 7);
        j = ((it - cg) / (D / 8)) * 8 + (lane >> 3) * 2;
    };
    // the warp's first kGItems items, decoded once (no divisions per tile)
    int it_c[kGItems], it_j[kGItems];
    // G_t items go to the worker warps (the MMA warp's item numbers start past them all)
    const int wbase = worker ? warp : (1 << 20);
#pragma unroll
    for (int i = 0; i < kGItems; ++i) item_cj(wbase + i * kMmaWarp, it_c[i], it_j[i]);
    auto g_at = [&](const TileIn& in, int c, int j, float& g0, float& g1) {
        const float* gp = a.grad + (int64_t)(in.b0 + j) * a.total_d + td.doff + c;
        g0 = j < in.nb ? __ldg(gp) : 0.f;
        g1 = j + 1 < in.nb ? __ldg(gp + a.total_d) : 0.f;
    };
    auto load_offsets = [&](int b0, TileIn& in) {
        in.b0 = b0;
        in.nb = tmin<int>(kDenseKT, bk1 - b0);
        in.q0 = __ldg(boff + b0);
        in.qend = __ldg(boff + b0 + in.nb);
        in.ol = __ldg(boff + b0 + tmin<int>(lane, in.nb));
    };
    auto load_inputs = [&](TileIn& in) {  // after load_offsets
#pragma unroll
        for (int kk = 0; kk < kDenseLk; ++kk) {
            const uint32_t q = in.q0 + (uint32_t)(perm + kk * kDenseWorkers);
            in.r[kk] = 0xffff;
            in.s[kk] = 0.f;
            if (worker && q < in.qend) {
                in.r[kk] = __ldg(ws.hrow + q);
                in.s[kk] = has_scale ? __ldg(ws.scale + q) : 1.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kGItems; ++i) {
            const int it = wbase + i * kMmaWarp;
            in.g[2 * i] = in.g[2 * i + 1] = 0.f;
            if (it < bitems) g_at(in, it_c[i], it_j[i], in.g[2 * i], in.g[2 * i + 1]);
        }
    };
    auto put_b = [&](int c, int j, int bb, float g0, float g1) {
        uint16_t t0[kDenseSplit], t1[kDenseSplit];
        split3(g0, t0);
        split3(g1, t1);
        const uint32_t off = core_off(c, j, sbo);
#pragma unroll
        for (int si = 0; si < kDenseSplit; ++si)
            *reinterpret_cast<uint32_t*>(Bs + (bb * kDenseSplit + si) * dense_b_bytes(D) + off) =
                (uint32_t)t0[si] | ((uint32_t)t1[si] << 16);
    };
    auto build_b = [&](const TileIn& in, int bb) {
#pragma unroll
        for (int i = 0; i < kGItems; ++i) {
            const int it = wbase + i * kMmaWarp;
            if (it < bitems) put_b(it_c[i], it_j[i], bb, in.g[2 * i], in.g[2 * i + 1]);
        }
        for (int it = wbase + kGItems * kMmaWarp; it < bitems; it += kMmaWarp) {
            int c, j;
            item_cj(it, c, j);
            float g0, g1;
            g_at(in, c, j, g0, g1);
            put_b(c, j, bb, g0, g1);
        }
    };

    // Histogram of a tile: the lookups of `in` (remembered in ent[kk]); the
    // rest (tiles of more than 2400 lookups) marks the tile `full`, whose
    // clears then cover whole arrays.
    // bag within the tile of each of its first 2400 lookups (16 threads per
    // bag), built two tiles ahead into one of two buffers
    auto build_tab = [&](const TileIn& in, int slot) {
        const int m = tid >> 4, sub = tid & 15;
        const uint32_t lo = __shfl_sync(0xffffffffu, in.ol, m);
        const uint32_t nx = __shfl_sync(0xffffffffu, in.ol, (m + 1) & 31);
        const uint32_t hi = m + 1 < in.nb ? nx : in.qend;
        if (m < in.nb)
            for (uint32_t q = lo + (uint32_t)sub; q < hi && q - in.q0 < (uint32_t)kDenseTab; q += 16)
                s_bagtab[slot][q - in.q0] = (uint8_t)m;
    };
    auto accumulate = [&](const TileIn& in, int slot, uint32_t(&ent)[kDenseLk], bool& full) {
        full = in.qend - in.q0 > (uint32_t)(kDenseWorkers * kDenseLk);
        auto one = [&](uint32_t q, int r, float sc, bool tab) -> uint32_t {
            if (!__any_sync(0xffffffffu, q < in.qend)) return kNoEntry;  // no lookup in this warp's slot
            // bag of q: from the table, else the last j < nb with first
            // lookup <= q (whole warp)
            int j = 0;
            if (tab) {
                if (q < in.qend) j = s_bagtab[slot][q - in.q0];
            } else {
#pragma unroll
                for (int step = 16; step > 0; step >>= 1) {
                    const uint32_t v = __shfl_sync(0xffffffffu, in.ol, j + step);
                    if (j + step < in.nb && v <= q) j += step;
                }
            }
            const int m = r - row0;
            if (q < in.qend && r < R && m >= 0 && m < Mp) {
                // the lookup that finds the entry empty owns it (writes and
                // clears its H^T terms); a sum that passes through zero can
                // make a second owner, which writes the same terms
                const float old = atomicAdd(&Hf[hf_index((uint32_t)m, (uint32_t)j)], sc);
                s_cnt[m] = 1u;  // the row is touched
                return old == 0.f ? (((uint32_t)m << 5) | (uint32_t)j) : kNoEntry;
            }
            return kNoEntry;
        };
#pragma unroll
        for (int kk = 0; kk < kDenseLk; ++kk)
            ent[kk] = one(worker ? in.q0 + (uint32_t)(perm + kk * kDenseWorkers) : 0xffffffffu, in.r[kk], in.s[kk],
                          true);
        if (full) {
            for (uint32_t base = in.q0 + kDenseWorkers * kDenseLk; base < in.qend; base += kDenseWorkers) {
                const uint32_t q = worker ? base + (uint32_t)perm : 0xffffffffu;
                int r = 0xffff;
                float sc = 0.f;
                if (q < in.qend) {
                    r = __ldg(ws.hrow + q);
                    sc = has_scale ? __ldg(ws.scale + q) : 1.f;
                }
                (void)one(q, r, sc, false);
            }
        }
    };

    uint32_t phase = 0;
    bool first = true, promoted = false, timed_out = false;
    const int lg = warp & 3;  // warp w reads tensor-memory lanes 32*(w%4) .. +31
    const uint32_t tlane = tmem + ((uint32_t)(lg * 32) << 16);
    // short accumulator (+ long sum so far) -> long sum; the short one restarts
    auto promote = [&]() {
        for (int i = 0; i < mtiles; ++i)
            for (int c = (warp >> 2) * 16; c < D; c += (kDenseWarps / 4) * 16) {
                float v[16];
                tmem_ld16(tlane + (uint32_t)(i * D + c), v);
                if (promoted) {
                    float u[16];
                    tmem_ld16(tlane + long0 + (uint32_t)(i * D + c), u);
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] += u[q];
                }
                tmem_st16(tlane + long0 + (uint32_t)(i * D + c), v);
            }
        tmem_st_wait();
        promoted = true;
        first = true;
    };

    uint32_t cur[kDenseLk], nxt[kDenseLk];
    bool full_cur = false, full_nxt = false;
#pragma unroll
    for (int kk = 0; kk < kDenseLk; ++kk) cur[kk] = nxt[kk] = kNoEntry;
    TileIn pf;  // inputs of the next tile to accumulate
    if (ntiles > 0) {
        load_offsets(bk0, pf);
        load_inputs(pf);
        build_tab(pf, 0);
        build_b(pf, 0);
        __syncthreads();  // the bag table
        accumulate(pf, 0, cur, full_cur);
        if (ntiles > 1) {
            load_offsets(bk0 + kDenseKT, pf);
            load_inputs(pf);
            build_tab(pf, 1);  // read after the loop's first syncs
        }
    }
    for (int kt = 0; kt < ntiles; ++kt) {
        const int buf = kt & 1;
        __syncthreads();  // histogram and G_t of this tile complete; last tile's H^T cleared
        // owned histogram entries -> H^T terms, the entry cleared for the
        // next tile (a zero sum leaves H^T's cleared entry as it is)
        if (!full_cur) {
#pragma unroll
            for (int kk = 0; kk < kDenseLk; ++kk) {
                if (cur[kk] == kNoEntry) continue;
                const uint32_t m = cur[kk] >> 5, j = cur[kk] & 31u;
                const float v = Hf[hf_index(m, j)];
                if (v == 0.f) continue;
                Hf[hf_index(m, j)] = 0.f;
                uint16_t tt[kDenseSplit];
                split3(v, tt);
                const uint32_t off = core_off((int)m, (int)j, sbo);
#pragma unroll
                for (int si = 0; si < kDenseSplit; ++si)
                    *reinterpret_cast<uint16_t*>(As + si * dense_a_bytes(Mp) + off) = tt[si];
            }
        } else {
            for (int e = tid; e < Mp * kDenseKT; e += kDenseThreads) {  // one thread per entry
                const uint32_t m = (uint32_t)e / kDenseKT, j = (uint32_t)e % kDenseKT;
                const float v = Hf[hf_index(m, j)];
                if (v == 0.f) continue;
                Hf[hf_index(m, j)] = 0.f;
                uint16_t tt[kDenseSplit];
                split3(v, tt);
                const uint32_t off = core_off((int)m, (int)j, sbo);
#pragma unroll
                for (int si = 0; si < kDenseSplit; ++si)
                    *reinterpret_cast<uint16_t*>(As + si * dense_a_bytes(Mp) + off) = tt[si];
            }
        }
        fence_proxy_async_smem();  // generic-proxy writes of A and B -> tensor cores
        tcgen05_before_sync();
        __syncthreads();
        tcgen05_after_sync();
        if (tid == kMmaWarp * 32) {
            // per M tile and K step, the six products x_i * y_j with i + j <= 2;
            // the first MMA of each M tile starts the sum after a restart
            const uint64_t bbuf = bdesc0 + (uint64_t)(buf * kDenseSplit) * b_split16;
            for (int i = 0; i < mtiles; ++i) {
#pragma unroll
                for (int ks = 0; ks < kDenseKT / 16; ++ks) {
                    const uint64_t a_ik = adesc0 + (uint64_t)(i * mtile16 + ks * kstep16);
                    const uint64_t b_k = bbuf + (uint64_t)(ks * kstep16);
                    const uint32_t d = tmem + (uint32_t)(i * D);
#pragma unroll
                    for (int pr = 0; pr < 6; ++pr) {
                        constexpr uint32_t kPa = 0x910, kPb = 0x184;  // (pa, pb): (0,0) (0,1) (1,0) (0,2) (1,1) (2,0)
                        const uint32_t pa = (kPa >> (2 * pr)) & 3u, pb = (kPb >> (2 * pr)) & 3u;
                        mma_f16(d, a_ik + (uint64_t)(pa * a_split16), b_k + (uint64_t)(pb * b_split16), idesc,
                                (first && ks == 0 && pr == 0) ? 0u : 1u);
                    }
                }
            }
            mma_commit(&s_bar);
        }
        first = false;
        // while the MMAs run: the next tile's histogram (cleared before the
        // sync above) and G_t from the prefetched inputs
        const bool more = kt + 1 < ntiles;
        if (more) {
            build_b(pf, buf ^ 1);
            accumulate(pf, buf ^ 1, nxt, full_nxt);
            if (kt + 2 < ntiles) load_offsets(bk0 + (kt + 2) * kDenseKT, pf);  // in flight during the wait
        }
        // every thread waits; the block agrees on the outcome
        const bool ok = mbar_wait(&s_bar, phase);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        phase ^= 1u;
        tcgen05_after_sync();
        if (more && kt + 2 < ntiles) {  // the tile after next: in flight from here on
            load_inputs(pf);
            build_tab(pf, buf);  // this tile's table is no longer read
        }
        // the MMAs have read H^T: clear what this tile wrote
        if (!full_cur) {
#pragma unroll
            for (int kk = 0; kk < kDenseLk; ++kk) {
                if (cur[kk] == kNoEntry) continue;
                const uint32_t off = core_off((int)(cur[kk] >> 5), (int)(cur[kk] & 31u), sbo);
#pragma unroll
                for (int si = 0; si < kDenseSplit; ++si)
                    *reinterpret_cast<uint16_t*>(As + si * dense_a_bytes(Mp) + off) = 0;
            }
        } else {
            uint4* pa = reinterpret_cast<uint4*>(As);
            const int n16 = (int)(kDenseSplit * dense_a_bytes(Mp) / 16);
            for (int i = tid; i < n16; i += kDenseThreads) pa[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        // each thread reads and writes only its own accumulator lanes and
        // columns; the syncs before the next MMAs order this before them
        if ((kt + 1) % kDensePromote == 0 || kt + 1 == ntiles) promote();
#pragma unroll
        for (int kk = 0; kk < kDenseLk; ++kk) cur[kk] = nxt[kk];
        full_cur = full_nxt;
    }
    if (!timed_out) {
        // long sum (zeros if the part had no bags) -> this part's gradient slice
        float* dg = ws.dgrad + (size_t)sp * a.total_floats + a.goff[k];
        for (int i = 0; i < mtiles; ++i) {
            const int r = row0 + i * 128 + lg * 32 + lane;
            for (int c = (warp >> 2) * 16; c < D; c += (kDenseWarps / 4) * 16) {
                float v[16];
                if (promoted) {
                    tmem_ld16(tlane + long0 + (uint32_t)(i * D + c), v);  // whole warp
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] = 0.f;
                }
                if (r < R) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<float4*>(dg + (int64_t)r * D + c)[q] =
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
        }
        __syncthreads();  // all touched-row flags in
        uint32_t* dc = ws.dcount + a.roff[k] + row0;
        for (int i = tid; i < rows_here; i += kDenseThreads)
            if (s_cnt[i]) dc[i] = 1u;  // touched (several parts store the same flag)
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
    chain_wait();  // returns at once unless launched chained
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

// The dense kernel's dynamic shared-memory limit, raised to the device's
// opt-in maximum less its static shared memory (on the current device; the
// attribute is per device).
cudaError_t dense_configure(int optin) {
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, dense_mma_kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dense_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    return e;
}

// Clears the touched-row flags, sums, updates (all on stream s).
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
    const unsigned grid = (unsigned)(a.n * groups_max * a.splits);
    dense_mma_kernel<<<grid, kDenseThreads, smem, s>>>(a, ws, groups_max);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned ublocks = (unsigned)((a.total_rows * 32 + 255) / 256);
    return launch_chained(dense_update_kernel, dim3(ublocks), dim3(256), s, a, ws);
}

}  // namespace tbe
