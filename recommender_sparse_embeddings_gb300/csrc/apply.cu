// Backward apply: per distinct (table,row) key, g = sum over its run of
// s_i * grad[bag_i, Doff_t : Doff_t + D_t] in fp32, then one optimizer update
// of that row (kimbodo "What Happened": one optimizer update per row, a
// streaming path for short runs, gradient accumulation for runs of at least
// 256 lookups).
//
// One kernel per backward class (table dtype x row shape) present in the
// handle, so each kernel's registers are sized for one shape only; the class
// kernels run side by side on the handle's apply streams.  A class kernel
// walks a work list table by table: the chunks of the table's long runs
// (numbered in key order by the preparation step; 256 to 1024 lookups, by
// batch size), then batches of up to kBatchRows consecutive distinct keys.
// Warps take work items from a per-class atomic counter.
//
// A sorted slot's value is the lookup's position when the batch has
// per-lookup scales (weights or mean pooling): its bag and scale are then
// read by position.  Without scales the sort carries the flat bag itself,
// which spares a random 4-byte read per lookup (from an N-entry array that
// on large batches does not stay in L2).
//
//  Short runs (fewer than kLongRun lookups), "streaming": a warp splits its
//    batch into pieces of at most R keys and walks each piece's sorted lookups
//    as one stream: sorted values, bags and scales are fetched 32 lookups at a
//    time one chunk ahead, gradient rows several at a time, and each lookup is
//    added to its key's sum.  The piece's table rows are read before the
//    stream starts so the read overlaps the gradient gather; after the stream
//    each key gets its optimizer step and its row is stored.  Sums are plain
//    fp32 (at most 255 terms).
//    Lanes own columns: a row is read by a group of LPR lanes (8 for dim 32,
//    16 for dim 64, 32 otherwise), lane l holding columns blk*LPR*4 +
//    (l%LPR)*4 + [0, 4) of each column block, so every gradient load is 16
//    bytes wide; the 32/LPR groups of a warp take different lookups of the
//    same keys and add their sums at the end.
//  Long runs, "accumulate": a warp sums one chunk of the run.  Every lane
//    takes the same lookup and holds VW = dim/32 consecutive columns, so one
//    load instruction reads a whole gradient row; G rows are loaded per step
//    (8 for dim <= 128, 2 for dim 256), and the chunk's sorted values, bags
//    and scales stream in 32 at a time, the bags and scales one window ahead
//    and the values two, so the gather never waits on its own metadata.  Each
//    step's G products are summed in fp32 (packed two-wide FMAs) and the
//    step sums added with compensated (Kahan) addition (consecutive lookups
//    of a long run often share a bag, so longer plain sums would round
//    coarsely); the partial row goes to the workspace.  The warp that
//    completes the last chunk of a run (atomic count after a fence) adds the
//    partials in chunk order with compensated addition, updates the row,
//    and resets the count so the prepared workspace can be applied again.
#include "tbe_internal.cuh"

namespace tbe {

// Distinct keys per short-run work item: 31 (every lane then holds a key's
// first slot, lane n the batch's end), or 16 when the batch would then give
// the apply warps fewer than sixteen items each (measured: the longer
// batches pay off on the hot-row workload, 23 items a warp, and lose on the
// mixed workload, 11).
constexpr int kBatchRows = 31;
constexpr int kBatchRowsSmall = 16;
// Resident CTAs of 256 threads per SM the class kernels are built for (80
// registers a thread); the grid is one wave of them.
constexpr int kApplyCtasPerSm = 3;

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


// Row shapes of the vector classes.  A row is read by a group of LPR lanes,
// each lane holding VW = 4 consecutive columns (16-byte gradient loads) of
// each of NB column blocks of LPR*4 columns; a warp holds NG = 32/LPR groups,
// which take different lookups of the same keys and add their sums up at the
// end.  Small rows thus still keep 16 bytes per lane in flight per load.
template <int CODE>
struct ShapeOf {
    static constexpr int VW = 4;
    static constexpr int LPR = CODE == SHAPE_D32 ? 8 : (CODE == SHAPE_D64 ? 16 : 32);
    static constexpr int NB = CODE == SHAPE_D256 ? 2 : 1;
    static constexpr int NG = 32 / LPR;
};

// ------------------------------------------------------- row slice helpers

// A lane's slice of one table row: NB blocks of VW consecutive elements,
// kept as raw 32-bit words (w[WORDS]) until needed.  Static helpers over a
// plain word array keep the slices in registers.
template <int DT, int VW, int NB, int LPR>
struct Slice {
    static constexpr int WPB = DT == DT_F32 ? VW : (VW + 1) / 2;  // words per block
    static constexpr int WORDS = WPB * NB;

    __device__ __forceinline__ static int col(int lane, int q) { return q * LPR * VW + (lane & (LPR - 1)) * VW; }

    __device__ __forceinline__ static void load(uint32_t (&w)[WORDS], const void* base, int64_t row, int dim,
                                                int lane) {
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            const int64_t k = row * dim + col(lane, q);
            if constexpr (DT == DT_F32) {
                const uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(base) + k);
                w[q * WPB + 0] = v.x; w[q * WPB + 1] = v.y; w[q * WPB + 2] = v.z; w[q * WPB + 3] = v.w;
            } else {
                const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(base) + k);
                w[q * WPB + 0] = v.x; w[q * WPB + 1] = v.y;
            }
        }
    }

    __device__ __forceinline__ static void store(const uint32_t (&w)[WORDS], void* base, int64_t row, int dim,
                                                 int lane) {
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            const int64_t k = row * dim + col(lane, q);
            if constexpr (DT == DT_F32)
                *reinterpret_cast<uint4*>(reinterpret_cast<float*>(base) + k) =
                    make_uint4(w[q * WPB], w[q * WPB + 1], w[q * WPB + 2], w[q * WPB + 3]);
            else
                *reinterpret_cast<uint2*>(reinterpret_cast<unsigned short*>(base) + k) =
                    make_uint2(w[q * WPB], w[q * WPB + 1]);
        }
    }

    __device__ __forceinline__ static float get(const uint32_t (&w)[WORDS], int q, int v) {
        if constexpr (DT == DT_F32) {
            return __uint_as_float(w[q * WPB + v]);
        } else {
            const uint32_t h = (w[q * WPB + v / 2] >> (16 * (v & 1))) & 0xffffu;
            return DT == DT_F16 ? h_bits_to_float(h) : bf16_bits_to_float(h);
        }
    }

    __device__ __forceinline__ static void set(uint32_t (&w)[WORDS], int q, int v, float x) {
        if constexpr (DT == DT_F32) {
            w[q * WPB + v] = __float_as_uint(x);
        } else {
            const uint32_t h = DT == DT_F16 ? (uint32_t)__half_as_ushort(__float2half_rn(x))
                                            : (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
            uint32_t& word = w[q * WPB + v / 2];
            word = (v & 1) ? ((word & 0x0000ffffu) | (h << 16)) : ((word & 0xffff0000u) | h);
        }
    }
};

// Loads the lane's 4 gradient floats starting at p.
__device__ __forceinline__ void ld_grad4(const float* p, float* f) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}

// Sums x over the NG row groups of the warp (butterfly over the lane bits
// above the group's own; every group ends with the same bits).
template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Optimizer step for one row given its gradient g (this lane's columns);
// `row` holds the old values and receives the new ones.  `m_old` is the row's
// Adagrad state (ignored by SGD); the new state is returned.  Every row group
// holding the same g computes the same result.
template <int DT, int VW, int NB, int LPR>
__device__ __forceinline__ float optimizer_step(const ApplyArgs& a, int dim, const float (&g)[NB][VW],
                                                uint32_t (&row)[Slice<DT, VW, NB, LPR>::WORDS], float m_old) {
    using S = Slice<DT, VW, NB, LPR>;
    if (a.opt == 2) {
        float sq = 0.f;
#pragma unroll
        for (int q = 0; q < NB; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v) sq = fmaf(g[q][v], g[q][v], sq);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        const float m = m_old + __fdiv_rn(sq, (float)dim);
        // lr / (sqrt(m) + eps) once per row (rounded once more than a
        // division per column)
        const float step = __fdiv_rn(a.lr, sqrtf(m) + a.eps);
#pragma unroll
        for (int q = 0; q < NB; ++q)
#pragma unroll
            for (int v = 0; v < VW; ++v) S::set(row, q, v, fmaf(-step, g[q][v], S::get(row, q, v)));
        return m;
    }
#pragma unroll
    for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int v = 0; v < VW; ++v) S::set(row, q, v, fmaf(-a.lr, g[q][v], S::get(row, q, v)));
    return m_old;
}

// ------------------------------------------------------------- short runs

// Metadata of 32 sorted lookups, lane k holding lookup w + k: b = bag row
// within the table (-1 past the batch's lookups or if the bag is out of
// range), s = scale.
struct Meta {
    int b;
    float s;
};

// Gradient rows in flight per row group (GROUP; NG*GROUP lookups per warp
// step, 2 KB of gradient per warp) and keys per piece (R), whose table-row
// slices and gradient sums stay in registers: R * (row words + columns) +
// GROUP * columns live words per lane, at most about 40.
template <int DT, int NB>
struct ShortTune {
    static constexpr int WORDS = Slice<DT, 4, NB, 32>::WORDS;
    static constexpr int COLS = 4 * NB;
    static constexpr int GROUP = 4 / NB;
    static constexpr int R0 = (40 - GROUP * COLS) / (WORDS + COLS);
    static constexpr int R = R0 > 8 ? 8 : (R0 < 1 ? 1 : R0);
};

__device__ __forceinline__ Meta load_meta(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                          uint32_t w, uint32_t Eend, int64_t tB, int lane) {
    const uint32_t i = w + lane;
    Meta m{-1, 1.f};
    if (i < Eend) {
        const uint32_t v = __ldg(sorted_val + i);  // position with scales, else the flat bag
        if (!a.has_scale || v < (uint32_t)a.N) {
            const uint32_t rel = (a.has_scale ? __ldg(ws.bag + v) : v) - (uint32_t)tB;
            if (rel < (uint32_t)a.B) m.b = (int)rel;
            if (a.has_scale) m.s = __ldg(ws.scale + v);
        }
    }
    return m;
}

// A sliding window over the batch's sorted lookups: metadata of lookups
// [w0, w0 + 64) in two 32-lookup halves; the next half is fetched as soon as
// the stream passes the middle, so it is in flight 32 lookups ahead.  (A
// deeper pipeline, positions two halves ahead, measured slower: the extra
// registers cost more than the waits it removes.)
struct MetaWindow {
    uint32_t w0;
    Meta m0, m1;
};

// One batch: distinct keys [u0, u0 + n) of table t (n <= kBatchRows).  Short
// keys are taken in pieces of at most R consecutive keys (a long or skipped
// key ends a piece, so a piece's lookups are exactly its keys' sorted slots);
// each piece's table rows are read first, then its lookups stream through
// the window, NG*GROUP per step (row group g takes lookups g, g + NG, ...),
// and each is added to its key's sum; the groups' sums are added up and each
// key gets its optimizer step.
template <int DT, int CODE>
__device__ __forceinline__ void short_batch_vec(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                                const TableDesc& td, int t, uint32_t rs, uint32_t key, float mstate,
                                                uint32_t rows, int lane) {
    using Sh = ShapeOf<CODE>;
    constexpr int VW = Sh::VW, NB = Sh::NB, LPR = Sh::LPR, NG = Sh::NG;
    using Tn = ShortTune<DT, NB>;
    using S = Slice<DT, VW, NB, LPR>;
    constexpr int R = Tn::R;
    constexpr int GROUP = Tn::GROUP;
    constexpr int WORDS = S::WORDS;
    constexpr int STEP = NG * GROUP;
    const int grp = lane / LPR;
    const int64_t tB = (int64_t)t * a.B;
    const int lastrow = 31 - __clz(rows);
    const uint32_t Eend = __shfl_sync(0xffffffffu, rs, lastrow + 1);

    MetaWindow win;
    win.w0 = 0xffffffffu;
    while (rows) {
        // the next piece: consecutive short keys [f, f + nk)
        const int f = __ffs(rows) - 1;
        int nk = 1;
#pragma unroll
        for (int k = 1; k < R; ++k)
            if (nk == k && ((rows >> (f + k)) & 1u)) nk = k + 1;
        rows &= ~(((1u << nk) - 1u) << f);
        const uint32_t E0 = __shfl_sync(0xffffffffu, rs, f);
        const uint32_t E1 = __shfl_sync(0xffffffffu, rs, f + nk);
        // first slots of the piece's later keys (a lookup's slot counts them)
        uint32_t pr[R];
#pragma unroll
        for (int k = 1; k < R; ++k) {
            const uint32_t x = __shfl_sync(0xffffffffu, rs, (f + k) & 31);
            pr[k] = k < nk ? x : 0xffffffffu;
        }

        // table rows of the piece (their loads overlap the stream below)
        uint32_t wrow[R][WORDS];
#pragma unroll
        for (int s = 0; s < R; ++s) {
            const uint32_t kr = __shfl_sync(0xffffffffu, key, (f + s) & 31);
            if (s < nk) S::load(wrow[s], td.data, (int64_t)kr - td.rowbase, td.dim, lane);
        }
        // window at the piece's first lookup
        if (win.w0 == 0xffffffffu || E0 < win.w0 || E0 >= win.w0 + 64) {
            win.w0 = E0;
            win.m0 = load_meta(a, ws, sorted_val, E0, Eend, tB, lane);
            win.m1 = load_meta(a, ws, sorted_val, E0 + 32, Eend, tB, lane);
        }
        float acc[R][NB][VW];
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int q = 0; q < NB; ++q)
#pragma unroll
                for (int v = 0; v < VW; ++v) acc[s][q][v] = 0.f;

        for (uint32_t i = E0; i < E1; i += STEP) {
            while (i >= win.w0 + 32) {  // slide: keep [w0, w0 + 64) ahead of i
                win.m0 = win.m1;
                win.w0 += 32;
                win.m1 = load_meta(a, ws, sorted_val, win.w0 + 32, Eend, tB, lane);
            }
            int sl[GROUP];
            float ss[GROUP];
            float g[GROUP][NB][VW];
#pragma unroll
            for (int u = 0; u < GROUP; ++u) {
                const uint32_t li = i + (uint32_t)(u * NG + grp);  // this group's lookup
                const uint32_t e = li - win.w0;                     // 0..63 (STEP <= 32)
                const int src = (int)(e & 31u);
                const bool hi = e >= 32u;
                const int b0 = __shfl_sync(0xffffffffu, win.m0.b, src);
                const int b1 = __shfl_sync(0xffffffffu, win.m1.b, src);
                const float s0 = __shfl_sync(0xffffffffu, win.m0.s, src);
                const float s1 = __shfl_sync(0xffffffffu, win.m1.s, src);
                const int b = hi ? b1 : b0;
                ss[u] = hi ? s1 : s0;
                int slot = 0;
#pragma unroll
                for (int k = 1; k < R; ++k) slot += pr[k] <= li ? 1 : 0;
                sl[u] = (li < E1 && b >= 0) ? slot : -1;
                const float* grow = a.grad + (int64_t)(b < 0 ? 0 : b) * a.total_d + td.doff;
#pragma unroll
                for (int q = 0; q < NB; ++q) {
                    if (sl[u] >= 0) {
                        ld_grad4(grow + S::col(lane, q), g[u][q]);
                    } else {
#pragma unroll
                        for (int v = 0; v < VW; ++v) g[u][q][v] = 0.f;
                    }
                }
            }
            // add each lookup to its key's sum (a select, not a branch, keeps
            // acc in registers)
#pragma unroll
            for (int u = 0; u < GROUP; ++u)
#pragma unroll
                for (int s = 0; s < R; ++s) {
                    const float w = sl[u] == s ? ss[u] : 0.f;
#pragma unroll
                    for (int q = 0; q < NB; ++q) {
                        ffma2(acc[s][q][0], acc[s][q][1], w, g[u][q][0], g[u][q][1]);
                        ffma2(acc[s][q][2], acc[s][q][3], w, g[u][q][2], g[u][q][3]);
                    }
                }
        }
        // one optimizer step per key of the piece; group 0 stores the rows
#pragma unroll
        for (int s = 0; s < R; ++s) {
            if (s < nk) {
                if constexpr (NG > 1) {
#pragma unroll
                    for (int q = 0; q < NB; ++q)
#pragma unroll
                        for (int v = 0; v < VW; ++v) acc[s][q][v] = group_sum<LPR>(acc[s][q][v]);
                }
                const int r = f + s;
                const uint32_t kr = __shfl_sync(0xffffffffu, key, r);
                const float m_old = __shfl_sync(0xffffffffu, mstate, r);
                const float mnew = optimizer_step<DT, VW, NB, LPR>(a, td.dim, acc[s], wrow[s], m_old);
                if (grp == 0) S::store(wrow[s], td.data, (int64_t)kr - td.rowbase, td.dim, lane);
                if (a.opt == 2 && lane == r) a.state[kr] = mnew;
            }
        }
    }
}

// Element-wise rows: one key at a time, whole warp, columns lane + 32*j of
// each 256-column block.  Adagrad needs the row's sum of squares before any
// column moves, so it makes two passes.  With partial_src, the gradient is
// the ordered sum of nchunks partial rows instead of the lookups [s0, s1).
template <int DT>
__device__ __forceinline__ void generic_row(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                            const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                                            const float* partial_src, uint32_t nchunks, int lane) {
    const int D = td.dim;
    const int64_t r = (int64_t)key - td.rowbase;
    const int64_t tB = (int64_t)t * a.B;
    float sq = 0.f;
    const int passes = a.opt == 2 ? 2 : 1;
    for (int pass = 0; pass < passes; ++pass) {
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
                for (uint32_t ch = 0; ch < nchunks; ++ch)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int c = cb + lane + 32 * j;
                        if (c < D) acc[j].add(__ldcg(partial_src + (int64_t)ch * a.part_stride + c));
                    }
            } else {
                for (uint32_t i = s0; i < s1; ++i) {
                    const uint32_t v = __ldg(sorted_val + i);  // position with scales, else the flat bag
                    if (a.has_scale && v >= (uint32_t)a.N) continue;
                    const int64_t bag = a.has_scale ? (int64_t)__ldg(ws.bag + v) : (int64_t)v;
                    if (bag < tB || bag >= tB + a.B) continue;
                    const float s = a.has_scale ? __ldg(ws.scale + v) : 1.f;
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
                const float w = load_elem<DT>(td.data, r * D + c);
                const float nw = a.opt == 2 ? w - a.lr * __fdiv_rn(g, denom) : fmaf(-a.lr, g, w);
                store_elem<DT>(td.data, r * D + c, nw);
            }
        }
        if (a.opt == 2 && pass == 1) {
            __syncwarp();
            if (lane == 0) a.state[key] = m;
        }
    }
}

// One batch: distinct keys [u0, u0 + n) of table t (n <= kBatchRows).
template <int DT, int CODE>
__device__ __forceinline__ void short_batch(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                            const TableDesc& td, int t, uint32_t u0, uint32_t n, int lane) {
    const uint32_t N = (uint32_t)a.N;
    // lane l <= n: first sorted slot of batch row l (lane n: end of the last
    // row); lanes past n hold N so no lookup maps to them
    uint32_t rs = N;
    if ((uint32_t)lane <= n) rs = tmin<uint32_t>(__ldg(ws.runstart + u0 + lane), N);
    uint32_t key = 0xffffffffu;
    if ((uint32_t)lane < n) key = __ldg(ws.uniq + u0 + lane);
    const uint32_t re = __shfl_down_sync(0xffffffffu, rs, 1);
    bool is_short = false;
    float mstate = 0.f;
    if ((uint32_t)lane < n && key < a.total_rows && re > rs && re - rs < (uint32_t)kLongRun) {
        is_short = true;
        if (a.opt == 2) mstate = a.state[key];
    }
    uint32_t rows = __ballot_sync(0xffffffffu, is_short);
    if constexpr (CODE == SHAPE_GENERIC) {
        while (rows) {
            const int r = __ffs(rows) - 1;
            rows &= rows - 1;
            const uint32_t kr = __shfl_sync(0xffffffffu, key, r);
            const uint32_t s0 = __shfl_sync(0xffffffffu, rs, r);
            const uint32_t s1 = __shfl_sync(0xffffffffu, rs, r + 1);
            generic_row<DT>(a, ws, sorted_val, td, t, kr, s0, s1, nullptr, 0, lane);
        }
    } else if (rows) {
        short_batch_vec<DT, CODE>(a, ws, sorted_val, td, t, rs, key, mstate, rows, lane);
    }
}

// ------------------------------------------------- long runs: row shapes

// A row is held by the whole warp, lane l holding columns [l*VW, l*VW + VW).
// G gradient rows are loaded per step (up to 4 KB a warp); PF partial rows
// are in flight when a long run's partials are added.
template <int CODE>
struct VecShape {
    static constexpr int D = CODE == SHAPE_D32 ? 32 : (CODE == SHAPE_D64 ? 64 : (CODE == SHAPE_D128 ? 128 : 256));
    static constexpr int VW = D / 32;
    static constexpr int G = VW == 8 ? 2 : (32 / VW > 8 ? 8 : 32 / VW);  // long runs
    static constexpr int PF = 32 / VW;
};

// VW gradient floats at p (4*VW bytes, aligned to min(16, 4*VW)).
template <int VW>
__device__ __forceinline__ void ld_gv(const float* p, float (&f)[VW]) {
    if constexpr (VW == 1) {
        f[0] = __ldg(p);
    } else if constexpr (VW == 2) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(p));
        f[0] = v.x; f[1] = v.y;
    } else {
#pragma unroll
        for (int h = 0; h < VW / 4; ++h) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p) + h);
            f[4 * h] = v.x; f[4 * h + 1] = v.y; f[4 * h + 2] = v.z; f[4 * h + 3] = v.w;
        }
    }
}

// The same through L2 only (partial rows written by other warps of this
// kernel).
template <int VW>
__device__ __forceinline__ void ld_gv_cg(const float* p, float (&f)[VW]) {
    if constexpr (VW == 1) {
        f[0] = __ldcg(p);
    } else if constexpr (VW == 2) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
        f[0] = v.x; f[1] = v.y;
    } else {
#pragma unroll
        for (int h = 0; h < VW / 4; ++h) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p) + h);
            f[4 * h] = v.x; f[4 * h + 1] = v.y; f[4 * h + 2] = v.z; f[4 * h + 3] = v.w;
        }
    }
}

template <int VW>
__device__ __forceinline__ void st_fv(float* p, const float (&f)[VW]) {
    if constexpr (VW == 1) {
        p[0] = f[0];
    } else if constexpr (VW == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
    } else {
#pragma unroll
        for (int h = 0; h < VW / 4; ++h)
            reinterpret_cast<float4*>(p)[h] = make_float4(f[4 * h], f[4 * h + 1], f[4 * h + 2], f[4 * h + 3]);
    }
}

// acc += s * x over VW columns (packed two-wide FMAs).
template <int VW>
__device__ __forceinline__ void fma_v(float (&acc)[VW], float s, const float (&x)[VW]) {
    if constexpr (VW == 1) {
        acc[0] = fmaf(s, x[0], acc[0]);
    } else {
#pragma unroll
        for (int v = 0; v < VW; v += 2) ffma2(acc[v], acc[v + 1], s, x[v], x[v + 1]);
    }
}

// A lane's VW consecutive elements of a table row, kept as raw 32-bit words.
template <int DT, int VW>
struct RowV {
    static constexpr int W = DT == DT_F32 ? VW : (VW + 1) / 2;

    // p: the lane's first element
    __device__ __forceinline__ static void load(uint32_t (&w)[W], const void* p) {
        if constexpr (DT == DT_F32) {
            if constexpr (VW == 1) {
                w[0] = *reinterpret_cast<const uint32_t*>(p);
            } else if constexpr (VW == 2) {
                const uint2 v = *reinterpret_cast<const uint2*>(p);
                w[0] = v.x; w[1] = v.y;
            } else {
#pragma unroll
                for (int h = 0; h < VW / 4; ++h) {
                    const uint4 v = reinterpret_cast<const uint4*>(p)[h];
                    w[4 * h] = v.x; w[4 * h + 1] = v.y; w[4 * h + 2] = v.z; w[4 * h + 3] = v.w;
                }
            }
        } else {
            if constexpr (VW == 1) {
                w[0] = *reinterpret_cast<const unsigned short*>(p);
            } else if constexpr (VW == 2) {
                w[0] = *reinterpret_cast<const uint32_t*>(p);
            } else if constexpr (VW == 4) {
                const uint2 v = *reinterpret_cast<const uint2*>(p);
                w[0] = v.x; w[1] = v.y;
            } else {
                const uint4 v = *reinterpret_cast<const uint4*>(p);
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            }
        }
    }

    __device__ __forceinline__ static void store(const uint32_t (&w)[W], void* p) {
        if constexpr (DT == DT_F32) {
            if constexpr (VW == 1) {
                *reinterpret_cast<uint32_t*>(p) = w[0];
            } else if constexpr (VW == 2) {
                *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
            } else {
#pragma unroll
                for (int h = 0; h < VW / 4; ++h)
                    reinterpret_cast<uint4*>(p)[h] = make_uint4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
            }
        } else {
            if constexpr (VW == 1) {
                *reinterpret_cast<unsigned short*>(p) = (unsigned short)(w[0] & 0xffffu);
            } else if constexpr (VW == 2) {
                *reinterpret_cast<uint32_t*>(p) = w[0];
            } else if constexpr (VW == 4) {
                *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
            } else {
                *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }

    __device__ __forceinline__ static float get(const uint32_t (&w)[W], int v) {
        if constexpr (DT == DT_F32) {
            return __uint_as_float(w[v]);
        } else {
            const uint32_t h = (w[v / 2] >> (16 * (v & 1))) & 0xffffu;
            return DT == DT_F16 ? h_bits_to_float(h) : bf16_bits_to_float(h);
        }
    }

    __device__ __forceinline__ static void set(uint32_t (&w)[W], int v, float x) {
        if constexpr (DT == DT_F32) {
            w[v] = __float_as_uint(x);
        } else {
            const uint32_t h = DT == DT_F16 ? (uint32_t)__half_as_ushort(__float2half_rn(x))
                                            : (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
            uint32_t& word = w[v / 2];
            word = (v & 1) ? ((word & 0x0000ffffu) | (h << 16)) : ((word & 0xffff0000u) | h);
        }
    }
};

// Optimizer step of one row held by the whole warp, given its gradient g
// (this lane's columns);
// `row` holds the old values and receives the new ones.  m_old: the row's
// Adagrad state (ignored by SGD); returns the new state.
template <int DT, int VW>
__device__ __forceinline__ float optimizer_step_w(const ApplyArgs& a, int dim, const float (&g)[VW],
                                                uint32_t (&row)[RowV<DT, VW>::W], float m_old) {
    using R = RowV<DT, VW>;
    if (a.opt == 2) {
        float sq = 0.f;
#pragma unroll
        for (int v = 0; v < VW; ++v) sq = fmaf(g[v], g[v], sq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        const float m = m_old + __fdiv_rn(sq, (float)dim);
        // lr / (sqrt(m) + eps) once per row (rounded once more than a
        // division per column)
        const float step = __fdiv_rn(a.lr, sqrtf(m) + a.eps);
#pragma unroll
        for (int v = 0; v < VW; ++v) R::set(row, v, fmaf(-step, g[v], R::get(row, v)));
        return m;
    }
#pragma unroll
    for (int v = 0; v < VW; ++v) R::set(row, v, fmaf(-a.lr, g[v], R::get(row, v)));
    return m_old;
}

// ------------------------------------------------- streaming the lookups

// Raw metadata of the sorted slot a lane looks ahead at, from its sorted
// value v: its flat bag (0xffffffff past the stream or for an invalid
// position) and its scale.  With scales (HS) v is a position and both are
// looked up; without, v is the bag itself.
template <bool HS>
__device__ __forceinline__ void meta_issue(const ApplyArgs& a, const Workspace& ws, uint32_t v, uint32_t& bag,
                                           float& s) {
    bag = 0xffffffffu;
    s = 0.f;
    if constexpr (HS) {
        if (v < (uint32_t)a.N) {
            bag = __ldg(ws.bag + v);
            s = __ldg(ws.scale + v);
        }
    } else {
        bag = v;
    }
}

__device__ __forceinline__ uint32_t val_issue(const uint32_t* sorted_val, uint32_t i, uint32_t end) {
    return i < end ? __ldg(sorted_val + i) : 0xffffffffu;
}

// The slots [E0, E1) of one table t as a stream of 32-slot windows.  Lane k
// holds, for the current window w, cb = bag row of slot w + k within the
// table (-1 if none) and cs = its scale; the next window's raw bag and scale
// and the sorted values of the one after are in flight meanwhile.
template <bool HS>
struct Stream {
    uint32_t p;     // sorted values of window w + 64
    uint32_t nbag;  // raw bags of window w + 32
    float ns;       // raw scales of window w + 32
    int cb;
    float cs;

    __device__ __forceinline__ void start(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                          uint32_t E0, uint32_t E1, int lane) {
        const uint32_t p0 = val_issue(sorted_val, E0 + lane, E1);
        meta_issue<HS>(a, ws, p0, nbag, ns);
        p = val_issue(sorted_val, E0 + 32 + lane, E1);
    }
    // Makes window w current and issues the loads of the two after it.
    __device__ __forceinline__ void advance(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                            uint32_t w, uint32_t E1, uint32_t tB, int lane) {
        const uint32_t rel = nbag - tB;
        cb = rel < (uint32_t)a.B ? (int)rel : -1;
        cs = cb < 0 ? 0.f : (HS ? ns : 1.f);
        meta_issue<HS>(a, ws, p, nbag, ns);
        p = val_issue(sorted_val, w + 64 + lane, E1);
    }
};

// Gradient rows of the lookups k0 .. k0+G-1 of the current window (those at
// or past n, or without a bag, read as zero rows).
template <int VW, int G, bool FULL>
__device__ __forceinline__ void load_step(const ApplyArgs& a, const float* gb, int cb, int k0, int n,
                                          float (&g)[G][VW]) {
#pragma unroll
    for (int u = 0; u < G; ++u) {
        const int k = k0 + u;
        const int b = __shfl_sync(0xffffffffu, cb, k & 31);
        if (FULL) {
            ld_gv<VW>(gb + (int64_t)b * a.total_d, g[u]);
        } else if (k < n && b >= 0) {
            ld_gv<VW>(gb + (int64_t)b * a.total_d, g[u]);
        } else {
#pragma unroll
            for (int v = 0; v < VW; ++v) g[u][v] = 0.f;
        }
    }
}

// The scale of lookup k of the current window (0 for one without a bag).
__device__ __forceinline__ float step_scale(float cs, int k) { return __shfl_sync(0xffffffffu, cs, k & 31); }

// ------------------------------------------------------------- long runs

// Partial sum of one chunk, sorted slots [s0, s1) of one key of table t:
// each step's G products summed in fp32, the step sums added with
// compensated addition (consecutive lookups of a long run often share a
// bag, so sums over many of them would grow and round coarsely); written to
// part_row.
template <int CODE, bool HS>
__device__ __forceinline__ void long_chunk_vec(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                               const TableDesc& td, int t, uint32_t s0, uint32_t s1, float* part_row,
                                               int lane) {
    using V = VecShape<CODE>;
    constexpr int VW = V::VW, G = V::G;
    const uint32_t tB = (uint32_t)t * (uint32_t)a.B;
    const float* gb = a.grad + td.doff + lane * VW;
    float sum[VW], cmp[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) sum[v] = cmp[v] = 0.f;
    // one step's sum into the compensated totals
    auto add_step = [&](const float (&blk)[VW]) {
        if constexpr (VW == 1) {
            Kahan k{sum[0], cmp[0]};
            k.add(blk[0]);
            sum[0] = k.s;
            cmp[0] = k.c;
        } else {
#pragma unroll
            for (int v = 0; v < VW; v += 2) kahan2(sum[v], sum[v + 1], cmp[v], cmp[v + 1], blk[v], blk[v + 1]);
        }
    };
    Stream<HS> st;
    st.start(a, ws, sorted_val, s0, s1, lane);
    for (uint32_t w = s0; w < s1; w += 32) {
        st.advance(a, ws, sorted_val, w, s1, tB, lane);
        const int n = (int)tmin<uint32_t>(32u, s1 - w);
        if (n == 32 && __all_sync(0xffffffffu, st.cb >= 0)) {
#pragma unroll 1
            for (int k0 = 0; k0 < 32; k0 += G) {
                float g[G][VW], blk[VW];
                load_step<VW, G, true>(a, gb, st.cb, k0, 32, g);
#pragma unroll
                for (int v = 0; v < VW; ++v) blk[v] = 0.f;
#pragma unroll
                for (int u = 0; u < G; ++u) fma_v<VW>(blk, HS ? step_scale(st.cs, k0 + u) : 1.f, g[u]);
                add_step(blk);
            }
        } else {
#pragma unroll 1
            for (int k0 = 0; k0 < n; k0 += G) {
                float g[G][VW], blk[VW];
                load_step<VW, G, false>(a, gb, st.cb, k0, n, g);
#pragma unroll
                for (int v = 0; v < VW; ++v) blk[v] = 0.f;
#pragma unroll
                for (int u = 0; u < G; ++u) fma_v<VW>(blk, HS ? step_scale(st.cs, k0 + u) : 1.f, g[u]);
                add_step(blk);
            }
        }
    }
    float x[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) x[v] = sum[v] - cmp[v];
    st_fv<VW>(part_row + lane * VW, x);
}

// The run's gradient: its nc partial rows added in chunk order (PF rows in
// flight, compensated addition), then the row's optimizer step.
template <int DT, int CODE>
__device__ __forceinline__ void long_combine_vec(const ApplyArgs& a, const TableDesc& td, uint32_t key,
                                                 const float* part0, uint32_t nc, int lane) {
    using V = VecShape<CODE>;
    constexpr int VW = V::VW, PF = V::PF;
    using R = RowV<DT, VW>;
    Kahan acc[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] = Kahan{0.f, 0.f};
    for (uint32_t j0 = 0; j0 < nc; j0 += PF) {
        float x[PF][VW];
#pragma unroll
        for (int k = 0; k < PF; ++k) {
            const uint32_t j = j0 + (uint32_t)k;
            ld_gv_cg<VW>(part0 + (int64_t)(j < nc ? j : 0) * a.part_stride + lane * VW, x[k]);
        }
#pragma unroll
        for (int k = 0; k < PF; ++k)
            if (j0 + (uint32_t)k < nc)
#pragma unroll
                for (int v = 0; v < VW; ++v) acc[v].add(x[k][v]);
    }
    float g[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) g[v] = acc[v].value();
    char* rp = static_cast<char*>(td.data) + ((int64_t)key - td.rowbase) * td.row_bytes +
               (int64_t)lane * VW * elem_bytes(DT);
    uint32_t row[R::W];
    R::load(row, rp);
    const float m_old = a.opt == 2 ? a.state[key] : 0.f;
    const float m = optimizer_step_w<DT, VW>(a, V::D, g, row, m_old);
    R::store(row, rp);
    if (a.opt == 2 && lane == 0) a.state[key] = m;
}


template <int DT, int CODE>
__device__ __forceinline__ void long_item(const ApplyArgs& a, const Workspace& ws, const uint32_t* sorted_val,
                                          const TableDesc& td, int t, uint32_t key, uint32_t s0, uint32_t s1,
                                          uint32_t chunk, uint32_t base, uint32_t nc, int lane) {
    float* part_row = ws.partial + (int64_t)chunk * a.part_stride;
    // 1) this chunk's partial sum
    if constexpr (CODE == SHAPE_GENERIC) {
        const int D = td.dim;
        const int64_t tB = (int64_t)t * a.B;
        for (int cb = 0; cb < D; cb += 256) {
            Kahan acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = Kahan{0.f, 0.f};
            for (uint32_t i = s0; i < s1; ++i) {
                const uint32_t v = __ldg(sorted_val + i);  // position with scales, else the flat bag
                if (a.has_scale && v >= (uint32_t)a.N) continue;
                const int64_t bag = a.has_scale ? (int64_t)__ldg(ws.bag + v) : (int64_t)v;
                if (bag < tB || bag >= tB + a.B) continue;
                const float s = a.has_scale ? __ldg(ws.scale + v) : 1.f;
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
    } else {
        if (a.has_scale)
            long_chunk_vec<CODE, true>(a, ws, sorted_val, td, t, s0, s1, part_row, lane);
        else
            long_chunk_vec<CODE, false>(a, ws, sorted_val, td, t, s0, s1, part_row, lane);
    }
    // 2) the warp that finishes a run's last chunk combines all of them
    __threadfence();
    __syncwarp();
    uint32_t done = 0;
    if (lane == 0) done = atomicAdd(ws.chunk_done + base, 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done != nc - 1) return;
    __threadfence();
    const float* part0 = ws.partial + (int64_t)base * a.part_stride;
    if constexpr (CODE == SHAPE_GENERIC)
        generic_row<DT>(a, ws, sorted_val, td, t, key, 0, 0, part0, nc, lane);
    else
        long_combine_vec<DT, CODE>(a, td, key, part0, nc, lane);
    // every chunk of this run has been counted: reset for the next apply call
    if (lane == 0) ws.chunk_done[base] = 0;
}

// ------------------------------------------------------------------ kernel

// All work of one backward class (table dtype DT, row shape CODE), table by
// table in key order: each class table's long-run chunks (one consecutive
// range cstart[t] .. cstart[t+1]), then its short-run batches of kb (16 or
// kBatchRows) distinct keys.  Neighbouring work items thus read gradient columns of the
// same table, which keeps them in L2.  Warps take items one at a time from an
// atomic counter, so no warp idles while work is left; the last warp to
// finish resets the counter, so apply can run again on the same prepared
// workspace.
template <int DT, int CODE>
__global__ void __launch_bounds__(256, kApplyCtasPerSm) apply_class_kernel(ApplyArgs a, Workspace ws, const uint32_t* sorted_val) {
    chain_wait();  // returns at once unless launched chained
    __shared__ uint32_t s_ibase[kMaxTables + 1];  // first work item of each class table
    __shared__ uint32_t s_warp[8];
    a.has_scale = ws.counters[CTR_HAS_SCALE] != 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t U = tmin<uint32_t>(*(volatile uint32_t*)&ws.counters[CTR_U], (uint32_t)a.N);
    const uint32_t nchunks =
        tmin<uint32_t>(*(volatile uint32_t*)&ws.counters[CTR_NCHUNK], (uint32_t)ws.max_chunks);
    const uint32_t N = (uint32_t)a.N;
    const uint32_t kb = U / kBatchRows >= 16u * gridDim.x * (blockDim.x >> 5) ? kBatchRows : kBatchRowsSmall;

    // work items (chunks + batches) of the class's tables, exclusive-scanned
    uint32_t carry = 0;
    for (int base = 0; base < a.class_count; base += 256) {
        const int k = base + threadIdx.x;
        uint32_t ni = 0;
        if (k < a.class_count) {
            const int t = a.class_tables[k];
            const uint32_t us = tmin<uint32_t>(__ldg(ws.ustart + t), U);
            const uint32_t ue = tmin<uint32_t>(tmax<uint32_t>(__ldg(ws.ustart + t + 1), us), U);
            const uint32_t cs = tmin<uint32_t>(__ldg(ws.cstart + t), nchunks);
            const uint32_t ce = tmin<uint32_t>(tmax<uint32_t>(__ldg(ws.cstart + t + 1), cs), nchunks);
            ni = (ce - cs) + (ue - us + kb - 1) / kb;
        }
        uint32_t x = ni;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        uint32_t before = 0, total = 0;
        for (int w = 0; w < 8; ++w) {
            if (w < warp) before += s_warp[w];
            total += s_warp[w];
        }
        if (k < a.class_count) s_ibase[k] = carry + before + x - ni;
        carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) s_ibase[a.class_count] = carry;
    __syncthreads();
    const uint32_t items = carry;

    for (;;) {
        uint32_t item = 0;
        if (lane == 0) item = atomicAdd(&ws.counters[CTR_WORK + a.cls], 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= items) break;
        int lo = 0, hi = a.class_count - 1;  // last class table with s_ibase <= item
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_ibase[mid] <= item)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int t = a.class_tables[lo];
        const TableDesc td = a.tabs[t];
        const uint32_t j = item - s_ibase[lo];
        const uint32_t cs = tmin<uint32_t>(__ldg(ws.cstart + t), nchunks);
        const uint32_t ce = tmin<uint32_t>(tmax<uint32_t>(__ldg(ws.cstart + t + 1), cs), nchunks);
        if (j < ce - cs) {
            // one chunk of a long run of this table
            const uint32_t g = cs + j;
            const uint2 e = __ldg(ws.chunk_info + g);
            const uint32_t u = e.x, g0 = e.y;
            if (u >= U || g < g0) continue;
            const uint32_t r0 = __ldg(ws.runstart + u);
            const uint32_t r1 = tmin<uint32_t>(__ldg(ws.runstart + u + 1), N);
            if (r1 <= r0) continue;
            const uint32_t chunk = (uint32_t)a.chunk;
            const uint32_t nc = (r1 - r0 + chunk - 1) / chunk;
            const uint32_t jc = g - g0;
            const uint32_t key = __ldg(ws.uniq + u);
            if (jc >= nc || g0 + nc > nchunks || key < (uint64_t)td.rowbase ||
                (uint64_t)key >= (uint64_t)td.rowbase + (uint64_t)td.rows)
                continue;
            const uint32_t s0 = r0 + jc * chunk;
            const uint32_t s1 = tmin<uint32_t>(s0 + chunk, r1);
            long_item<DT, CODE>(a, ws, sorted_val, td, t, key, s0, s1, g, g0, nc, lane);
        } else {
            const uint32_t us = tmin<uint32_t>(__ldg(ws.ustart + t), U);
            const uint32_t ue = tmin<uint32_t>(tmax<uint32_t>(__ldg(ws.ustart + t + 1), us), U);
            const uint32_t u0 = us + (j - (ce - cs)) * kb;
            if (u0 >= ue) continue;
            short_batch<DT, CODE>(a, ws, sorted_val, td, t, u0, tmin<uint32_t>(kb, ue - u0), lane);
        }
    }
    // every warp has taken its last item: the last one to leave resets the
    // counters for the next apply call on this workspace
    if (lane == 0) {
        const uint32_t total_warps = gridDim.x * (blockDim.x >> 5);
        const uint32_t done = atomicAdd(&ws.counters[CTR_EXIT + a.cls], 1u);
        if (done == total_warps - 1) {
            atomicExch(&ws.counters[CTR_WORK + a.cls], 0u);
            atomicExch(&ws.counters[CTR_EXIT + a.cls], 0u);
        }
    }
}

template <int DT, int CODE>
static cudaError_t launch_class(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos, unsigned grid,
                                cudaStream_t s, bool chained) {
    if (chained) return launch_chained(apply_class_kernel<DT, CODE>, dim3(grid), dim3(256), s, a, ws, pos);
    apply_class_kernel<DT, CODE><<<grid, 256, 0, s>>>(a, ws, pos);
    return cudaGetLastError();
}

// chained: another class kernel of this call runs just before on stream s
template <int DT>
static cudaError_t launch_dtype(const ApplyArgs& a, const Workspace& ws, const uint32_t* pos, int code,
                                unsigned grid, cudaStream_t s, bool chained) {
    switch (code) {
        case SHAPE_D32: return launch_class<DT, SHAPE_D32>(a, ws, pos, grid, s, chained);
        case SHAPE_D64: return launch_class<DT, SHAPE_D64>(a, ws, pos, grid, s, chained);
        case SHAPE_D128: return launch_class<DT, SHAPE_D128>(a, ws, pos, grid, s, chained);
        case SHAPE_D256: return launch_class<DT, SHAPE_D256>(a, ws, pos, grid, s, chained);
        default: return launch_class<DT, SHAPE_GENERIC>(a, ws, pos, grid, s, chained);
    }
}

cudaError_t launch_apply(const ApplyArgs& a_in, const Workspace& ws, const int32_t* class_tables,
                         const int* class_begin, const int* class_count, const DenseArgs* dense,
                         cudaStream_t s, const cudaStream_t* streams, cudaEvent_t ev_fork,
                         const cudaEvent_t* ev_join) {
    if (a_in.N == 0) return cudaSuccess;
    const uint32_t* sorted_val = ws.vals[ws.sorted_buf];
    const unsigned grid = (unsigned)(a_in.num_sms * kApplyCtasPerSm);
    int present = dense ? 1 : 0;  // the dense tables' work counts as one more launch group
    for (int cls = 0; cls < kNumClasses; ++cls) present += class_count[cls] > 0;
    // more than one group: fork onto the side streams, which start after
    // everything already queued on s
    const bool fork = present > 1;
    if (fork) {
        cudaError_t e = cudaEventRecord(ev_fork, s);
        for (int i = 0; i < kApplyStreams && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(streams[i], ev_fork, 0);
        if (e != cudaSuccess) return e;
    }
    int k = 0;
    if (dense) {
        const cudaError_t e = launch_dense(*dense, ws, fork ? streams[k % kApplyStreams] : s);
        ++k;
        if (e != cudaSuccess) return e;
    }
    for (int cls = 0; cls < kNumClasses; ++cls) {
        if (class_count[cls] == 0) continue;
        ApplyArgs a = a_in;
        a.cls = cls;
        a.class_tables = class_tables + class_begin[cls];
        a.class_count = class_count[cls];
        const int dt = cls / NUM_SHAPES;
        // an unaligned gradient buffer rules out vector loads: element-wise
        const int code = a.grad_vec ? cls % NUM_SHAPES : SHAPE_GENERIC;
        cudaStream_t cs = fork ? streams[k % kApplyStreams] : s;
        const bool chained = fork && k >= kApplyStreams;  // the stream ran a group of this call already
        ++k;
        cudaError_t e;
        if (dt == DT_F32)
            e = launch_dtype<DT_F32>(a, ws, sorted_val, code, grid, cs, chained);
        else if (dt == DT_F16)
            e = launch_dtype<DT_F16>(a, ws, sorted_val, code, grid, cs, chained);
        else
            e = launch_dtype<DT_BF16>(a, ws, sorted_val, code, grid, cs, chained);
        if (e != cudaSuccess) return e;
    }
    if (fork) {
        // join: s waits for every side stream
        for (int i = 0; i < kApplyStreams; ++i) {
            cudaError_t e = cudaEventRecord(ev_join[i], streams[i]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_join[i], 0);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace tbe
