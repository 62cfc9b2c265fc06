// C ABI of the TBE library: argument checks, the handle's descriptor block,
// the backward workspace layout, and the order of kernel launches.  The
// declarations and their contracts are in include/tbe.h.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/tbe.h"
#include "tbe_internal.cuh"

namespace tbe {
cudaError_t launch_forward_schedule(TableDesc* tabs, int T, int B, cudaStream_t s);
}

using namespace tbe;

struct tbe_handle {
    int device = 0;
    int T = 0;
    int pooling = 0;
    uint32_t flags = 0;
    int num_sms = 0;
    std::vector<TableDesc> tabs;
    void* dev = nullptr;          // DevBlock, TableDesc[T], class table list[T]
    DevBlock* blk = nullptr;
    TableDesc* dtabs = nullptr;
    int32_t* dclass_tables = nullptr;
    int32_t* dhist_tables = nullptr;  // histogram-path tables: f16 ones, then bf16 ones
    HistGroup hist_f16{}, hist_bf16{};
    // dense-backward tables (the histogram tables unless TBE_FLAG_SORTED_BACKWARD)
    int n_dense = 0;
    int32_t* ddense_tables = nullptr;   // device [n_dense]
    int64_t* ddense_goff = nullptr;     // device [n_dense+1]: first gradient float of each
    int64_t* ddense_roff = nullptr;     // device [n_dense+1]: first row count of each
    int64_t dense_floats = 0, dense_rows = 0;
    int dense_max_rows = 0, dense_max_dim = 0;
    int dense_groups = 1;               // CTAs per table for its rows (128-row tiles per CTA)
    int class_begin[kNumClasses] = {};
    int class_count[kNumClasses] = {};
    int total_d = 0;
    int max_dim = 0;
    uint64_t total_rows = 0;
    int key_bits = 1;
    int digit_bits = 8;
    int passes = 1;
    int last_B = -1;
    int parity = 0;
    // the forward's length-keyed bag order: counts [T][kLenBuckets], flags
    // [T], CTA counters [T], order [T][B]; grown when a batch needs more
    void* dorder = nullptr;
    int64_t order_cap = 0;  // bags (T x B) the order array holds
    int vec_out = 0;
    cudaStream_t side = nullptr;  // preparation stream of tbe_forward_prepare
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    // streams the backward class kernels run on side by side
    cudaStream_t apply_streams[kApplyStreams] = {};
    cudaEvent_t ev_apply_fork = nullptr;
    cudaEvent_t ev_apply_join[kApplyStreams] = {};
};

namespace {

// A named NVTX range around one ABI call, so a profiler's timeline shows
// which call queued which kernels (a no-op unless a tool is attached).
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
size_t tabs_offset() { return align_up(sizeof(DevBlock)); }
size_t class_list_offset(int T) { return align_up(tabs_offset() + sizeof(TableDesc) * T); }
size_t hist_list_offset(int T) { return align_up(class_list_offset(T) + sizeof(int32_t) * T); }
size_t dense_list_offset(int T) { return align_up(hist_list_offset(T) + sizeof(int32_t) * T); }
size_t dense_off_offset(int T) { return align_up(dense_list_offset(T) + sizeof(int32_t) * T); }
size_t dev_block_bytes(int T) { return dense_off_offset(T) + 2 * sizeof(int64_t) * (T + 1); }

// Small tables the tensor-core histogram path can take: 16-bit rows whose
// dim is a multiple of 16 in [16, 256] (the MMA's N), 16-byte aligned data,
// at most max_rows rows (the MMA's K, padded to 16).  Whether its A operand
// and W^T fit one CTA's shared memory next to the other tables of its dtype
// is checked when the group is formed.
bool hist_eligible(const TableDesc& d, int64_t max_rows) {
    if (d.dtype != TBE_F16 && d.dtype != TBE_BF16) return false;
    if (d.dim % 16 != 0 || d.dim < 16 || d.dim > 256) return false;
    if (((uintptr_t)d.data % 16) != 0) return false;
    return d.rows <= max_rows;
}

// Adds table d to a histogram group if the group's shared memory (with 1 KB
// for the kernel's static arrays, about 0.8 KB) still fits `limit`.
bool hist_join(HistGroup& g, const TableDesc& d, size_t limit) {
    const int kp = (int)((d.rows + 63) & ~int64_t(63));
    const int kmax = std::max(g.kmax, kp);
    const size_t wt = std::max(g.wt_bytes, (size_t)d.dim * kp * 2);
    const size_t smem = hist_smem_bytes(kmax, wt);
    if (smem + 1024 > limit) return false;
    g.kmax = kmax;
    g.wt_bytes = wt;
    g.smem = smem;
    g.dmax = std::max(g.dmax, (int)d.dim);
    ++g.n;
    return true;
}

// Backward class of a table: dtype and row shape (vector lanes for dim 32,
// 64, 128, 256 when rows and gradient columns are 16-byte aligned, which the
// vector classes' 16-byte gradient loads need).
int backward_class(const TableDesc& d, int total_d) {
    const bool rows16 = ((uintptr_t)d.data % 16) == 0;
    const bool a4 = rows16 && d.doff % 4 == 0 && total_d % 4 == 0;
    int shape = SHAPE_GENERIC;
    if (a4) {
        if (d.dim == 32)
            shape = SHAPE_D32;
        else if (d.dim == 64)
            shape = SHAPE_D64;
        else if (d.dim == 128)
            shape = SHAPE_D128;
        else if (d.dim == 256)
            shape = SHAPE_D256;
    }
    return d.dtype * NUM_SHAPES + shape;
}

int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Parts each dense table's bags are split into for a batch of B bags (one
// CTA and one gradient slice each; one CTA per SM): the count of at most 8
// that best fills whole waves, with at least 64 bags per part.
int dense_parts(const tbe_handle* h, int64_t B) {
    if (h->n_dense == 0) return 1;
    const int64_t ctas = (int64_t)h->n_dense * h->dense_groups;
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 8 && (s == 1 || B / s >= 64); ++s) {
        const double waves = (double)((ctas * s + h->num_sms - 1) / h->num_sms);
        const double cost = waves / s;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Floats per partial-sum row: the widest dim rounded up to 16 bytes, so the
// vector classes read partial rows with 16-byte loads.
int part_stride(const tbe_handle* h) { return (h->max_dim + 3) / 4 * 4; }

struct Layout {
    size_t counters, hist, tile_bag, tcount, keys0, keys1, vals0, vals1, bag, scale, uniq, runstart,
        chunk_info, chunk_done, cstart, ustart, tpos, cbase, hrow, dboff, dgrad, dcount, partial, total;
    size_t zero_bytes;  // counters..tile_bag are zeroed per call
    int64_t max_chunks;
    int tiles;
};

Layout make_layout(const tbe_handle* h, int64_t N, int64_t B, bool scale) {
    Layout L{};
    const int64_t n = std::max<int64_t>(N, 1);
    L.tiles = (int)((N + kSortTile - 1) / kSortTile);
    L.max_chunks = 2 * (N / kLongRun) + 2;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes);
        return at;
    };
    L.counters = take(sizeof(uint32_t) * CTR_COUNT);
    L.hist = take(sizeof(uint32_t) * kMaxPasses * kMaxRadix);
    L.tile_bag = take(sizeof(uint32_t) * std::max(L.tiles, 1));
    L.zero_bytes = o;
    L.tcount = take(sizeof(uint32_t) * std::max(L.tiles, 1) * ((size_t)1 << h->digit_bits));
    L.keys0 = take(sizeof(uint32_t) * n);
    L.keys1 = take(sizeof(uint32_t) * n);
    L.vals0 = take(sizeof(uint32_t) * n);
    L.vals1 = take(sizeof(uint32_t) * n);
    L.bag = take(sizeof(uint32_t) * n);
    L.scale = scale ? take(sizeof(float) * n) : 0;
    L.uniq = take(sizeof(uint32_t) * n);
    L.runstart = take(sizeof(uint32_t) * (n + 1));
    L.chunk_info = take(sizeof(uint2) * L.max_chunks);
    L.chunk_done = take(sizeof(uint32_t) * L.max_chunks);
    L.cstart = take(sizeof(uint32_t) * (h->T + 1));
    L.ustart = take(sizeof(uint32_t) * (h->T + 1));
    L.tpos = take(sizeof(uint32_t) * (h->T + 1));
    L.cbase = take(sizeof(uint32_t) * (h->T + 1));
    if (h->n_dense > 0) {
        L.hrow = take(sizeof(uint16_t) * n);
        L.dboff = take(sizeof(uint32_t) * (size_t)h->n_dense * (size_t)(std::max<int64_t>(B, 0) + 1));
        L.dgrad = take(sizeof(float) * (size_t)h->dense_floats * dense_parts(h, B));
        L.dcount = take(sizeof(uint32_t) * (size_t)h->dense_rows);
    }
    L.partial = take(sizeof(float) * (size_t)L.max_chunks * part_stride(h));
    L.total = o;
    return L;
}

bool needs_scale(const tbe_handle* h, const float* weights) {
    return weights != nullptr || h->pooling == TBE_POOL_MEAN;
}

Workspace bind(const tbe_handle* h, const Layout& L, void* base, bool scale) {
    char* p = static_cast<char*>(base);
    Workspace w{};
    w.counters = reinterpret_cast<uint32_t*>(p + L.counters);
    w.hist = reinterpret_cast<uint32_t*>(p + L.hist);
    w.tcount = reinterpret_cast<uint32_t*>(p + L.tcount);
    w.tile_bag = reinterpret_cast<uint32_t*>(p + L.tile_bag);
    w.keys[0] = reinterpret_cast<uint32_t*>(p + L.keys0);
    w.keys[1] = reinterpret_cast<uint32_t*>(p + L.keys1);
    w.vals[0] = reinterpret_cast<uint32_t*>(p + L.vals0);
    w.vals[1] = reinterpret_cast<uint32_t*>(p + L.vals1);
    w.bag = reinterpret_cast<uint32_t*>(p + L.bag);
    w.scale = scale ? reinterpret_cast<float*>(p + L.scale) : nullptr;
    w.uniq = reinterpret_cast<uint32_t*>(p + L.uniq);
    w.runstart = reinterpret_cast<uint32_t*>(p + L.runstart);
    w.chunk_info = reinterpret_cast<uint2*>(p + L.chunk_info);
    w.chunk_done = reinterpret_cast<uint32_t*>(p + L.chunk_done);
    w.cstart = reinterpret_cast<uint32_t*>(p + L.cstart);
    w.ustart = reinterpret_cast<uint32_t*>(p + L.ustart);
    w.tpos = reinterpret_cast<uint32_t*>(p + L.tpos);
    w.cbase = reinterpret_cast<uint32_t*>(p + L.cbase);
    w.compact = h->n_dense > 0;
    if (w.compact) {
        w.hrow = reinterpret_cast<uint16_t*>(p + L.hrow);
        w.dboff = reinterpret_cast<uint32_t*>(p + L.dboff);
        w.dgrad = reinterpret_cast<float*>(p + L.dgrad);
        w.dcount = reinterpret_cast<uint32_t*>(p + L.dcount);
    }
    w.partial = reinterpret_cast<float*>(p + L.partial);
    w.max_chunks = L.max_chunks;
    w.tiles = L.tiles;
    w.passes = h->passes;
    w.digit_bits = h->digit_bits;
    // the sort ping-pongs once per pass, starting from buffer 0
    w.sorted_buf = h->passes % 2;
    return w;
}

// The scale array exists whenever weights or mean pooling are in play; the
// workspace is always laid out with room for it so its size only depends on
// the batch shape.
constexpr bool kLayoutWithScale = true;

// The handle's kernels, streams and descriptor block belong to the device
// that was current at tbe_create; a call made with another device current
// is refused before anything launches.
bool on_handle_device(const tbe_handle* h) {
    int d = -1;
    return cudaGetDevice(&d) == cudaSuccess && d == h->device;
}

int check_batch(const tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                int64_t N, int32_t B) {
    if (!h) return TBE_ERR_INVALID_ARG;
    if (!on_handle_device(h)) return TBE_ERR_INVALID_ARG;
    if (index_dtype != TBE_I32 && index_dtype != TBE_I64) return TBE_ERR_INVALID_ARG;
    if (N < 0 || B < 0) return TBE_ERR_INVALID_ARG;
    if (N >= (int64_t(1) << 30)) return TBE_ERR_UNSUPPORTED;
    if ((int64_t)h->T * B >= (int64_t(1) << 31)) return TBE_ERR_UNSUPPORTED;
    if (!offsets) return TBE_ERR_INVALID_ARG;
    if (N > 0 && !indices) return TBE_ERR_INVALID_ARG;
    if (B == 0 && N > 0) return TBE_ERR_INVALID_ARG;
    return TBE_OK;
}

// The last failing CUDA call of this host thread, for tbe_last_cuda_error.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = e;
    return TBE_ERR_CUDA;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? TBE_OK : cuda_fail(e); }

// Device bytes of the length-keyed order for n = T x B bags.
size_t order_bytes(const tbe_handle* h, int64_t n) {
    return sizeof(uint32_t) * ((size_t)h->T * (kLenBuckets + 2) + (size_t)n);
}

// With TBE_FLAG_LENGTH_ORDER: the order arrays, grown for T x B bags.
int ensure_order(tbe_handle* h, int32_t B) {
    const int64_t n = (int64_t)h->T * B;
    if ((h->flags & TBE_FLAG_LENGTH_ORDER) && n > h->order_cap) {
        // grow the order array (cudaFree waits for the device: no kernel
        // still reads the old one)
        if (h->dorder) cudaFree(h->dorder);
        h->dorder = nullptr;
        h->order_cap = 0;
        const cudaError_t e = cudaMalloc(&h->dorder, order_bytes(h, n));
        if (e != cudaSuccess) {
            h->dorder = nullptr;
            return e == cudaErrorMemoryAllocation ? TBE_ERR_NO_MEMORY : cuda_fail(e);
        }
        // the counts and the per-table CTA counters start at zero (the
        // kernels leave them so)
        const cudaError_t z = cudaMemset(h->dorder, 0, order_bytes(h, 0));
        if (z != cudaSuccess) return cuda_fail(z);
        h->order_cap = n;
    }
    return TBE_OK;
}

// Order arrays and the forward's warp map for batch size B.
int ensure_schedule(tbe_handle* h, int32_t B, cudaStream_t s) {
    const int rc = ensure_order(h, B);
    if (rc) return rc;
    if (B == h->last_B) return TBE_OK;
    cudaError_t e = launch_forward_schedule(h->dtabs, h->T, B, s);
    if (e != cudaSuccess) return cuda_fail(e);
    h->last_B = B;
    return TBE_OK;
}

}  // namespace

extern "C" {

int tbe_create(const tbe_table* tables, int32_t num_tables, int32_t pooling, uint32_t flags,
               tbe_handle** out) {
    CallRange range("tbe_create");
    if (!out) return TBE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!tables || num_tables <= 0) return TBE_ERR_INVALID_ARG;
    if (num_tables > kMaxTables) return TBE_ERR_UNSUPPORTED;
    if (pooling != TBE_POOL_SUM && pooling != TBE_POOL_MEAN) return TBE_ERR_INVALID_ARG;
    if (flags & ~(TBE_FLAG_NO_HISTOGRAM | TBE_FLAG_FORCE_HISTOGRAM | TBE_FLAG_SORTED_BACKWARD | TBE_FLAG_LENGTH_ORDER))
        return TBE_ERR_INVALID_ARG;
    tbe_handle* h = new (std::nothrow) tbe_handle();
    if (!h) return TBE_ERR_NO_MEMORY;
    h->T = num_tables;
    h->pooling = pooling;
    h->flags = flags;
    h->tabs.resize(num_tables);
    int64_t rowbase = 0;
    int doff = 0;
    bool vec_cols = true;
    for (int t = 0; t < num_tables; ++t) {
        const tbe_table& in = tables[t];
        if (in.rows <= 0 || in.dim <= 0 || !in.data) {
            delete h;
            return TBE_ERR_INVALID_ARG;
        }
        if (in.dtype != TBE_F32 && in.dtype != TBE_F16 && in.dtype != TBE_BF16) {
            delete h;
            return TBE_ERR_INVALID_ARG;
        }
        if (in.rows >= (int64_t(1) << 31) || in.dim > 4096) {
            delete h;
            return TBE_ERR_UNSUPPORTED;
        }
        TableDesc& d = h->tabs[t];
        std::memset(&d, 0, sizeof d);
        d.data = in.data;
        d.rows = in.rows;
        d.rowbase = rowbase;
        d.dim = in.dim;
        d.doff = doff;
        d.dtype = in.dtype;
        d.row_bytes = in.dim * elem_bytes(in.dtype);
        const int nvec = d.row_bytes / 16;
        const bool vec = d.row_bytes % 16 == 0 && ((uintptr_t)in.data % 16) == 0 && nvec <= 128;
        if (vec) {
            d.path = PATH_VEC;
            d.lanes = next_pow2(std::min(nvec, 32));
            d.vecs = (nvec + 31) / 32;  // column blocks of 32 vectors, one warp each
        } else {
            d.path = PATH_SCALAR;
            d.lanes = 32;
            d.vecs = 1;
        }
        if (doff % 4 != 0) vec_cols = false;
        rowbase += in.rows;
        doff += in.dim;
        h->max_dim = std::max(h->max_dim, (int)in.dim);
    }
    if ((uint64_t)rowbase >= 0xffffffffull) {
        delete h;
        return TBE_ERR_UNSUPPORTED;
    }
    h->total_rows = (uint64_t)rowbase;
    h->total_d = doff;
    h->vec_out = vec_cols && (doff % 4 == 0);
    int bits = 1;
    while (bits < 32 && (uint64_t(1) << bits) <= h->total_rows) ++bits;  // values 0..total_rows
    h->key_bits = bits;
    // 8-bit digits, or 9-bit ones when they save a pass
    h->digit_bits = (bits + kMaxRadixBits - 1) / kMaxRadixBits < (bits + kRadixBits - 1) / kRadixBits
                        ? kMaxRadixBits
                        : kRadixBits;
    h->passes = (bits + h->digit_bits - 1) / h->digit_bits;

    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e);
    }
    std::vector<int32_t> hist_f16, hist_bf16;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
    // the tensor-core kernels may use up to the opt-in shared memory on this
    // device (the limit is a per-device attribute of each kernel)
    if (e == cudaSuccess) e = hist_configure(optin);
    if (e == cudaSuccess) e = dense_configure(optin);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e);
    }
    // Small tables (hist_eligible: 16-bit rows, dim a multiple of 16 up to
    // 256, at most 512 rows, or 1024 with TBE_FLAG_FORCE_HISTOGRAM) take the
    // dense tensor-core backward unless TBE_FLAG_SORTED_BACKWARD; their
    // forward takes the histogram tensor-core path only with
    // TBE_FLAG_FORCE_HISTOGRAM (and when their dtype's group fits one CTA's
    // shared memory), the gather otherwise: measured on the 64 fp16 512 x 64
    // tables of the small-table workload, the gather pools them in 1.38 ms
    // and the histogram path in 2.07 ms, while the dense backward takes their
    // preparation from 2.31 to 0.71 ms.  TBE_FLAG_NO_HISTOGRAM turns both off.
    std::vector<char> small(num_tables, 0);
    if (!(flags & TBE_FLAG_NO_HISTOGRAM)) {
        const int64_t max_rows = (flags & TBE_FLAG_FORCE_HISTOGRAM) ? 1024 : 512;
        for (int t = 0; t < num_tables; ++t) {
            TableDesc& d = h->tabs[t];
            if (!hist_eligible(d, max_rows)) continue;
            small[t] = 1;
            if (!(flags & TBE_FLAG_FORCE_HISTOGRAM)) continue;
            HistGroup& g = d.dtype == TBE_F16 ? h->hist_f16 : h->hist_bf16;
            if (!hist_join(g, d, (size_t)optin)) continue;
            d.path = PATH_HIST;
            (d.dtype == TBE_F16 ? hist_f16 : hist_bf16).push_back(t);
        }
    }
    // dense backward: the small tables, unless the sorted path is asked for
    std::vector<int32_t> dense;
    std::vector<int64_t> dense_off;  // goff[0..n], then roff[0..n]
    {
        std::vector<int64_t> goff{0}, roff{0};
        for (int t = 0; t < num_tables; ++t) {
            TableDesc& d = h->tabs[t];
            d.dslot = -1;
            if (!small[t] || (flags & TBE_FLAG_SORTED_BACKWARD)) continue;
            d.dslot = (int32_t)dense.size();
            dense.push_back(t);
            goff.push_back(goff.back() + d.rows * d.dim);
            roff.push_back(roff.back() + d.rows);
            h->dense_max_rows = std::max(h->dense_max_rows, (int)d.rows);
            h->dense_max_dim = std::max(h->dense_max_dim, (int)d.dim);
        }
        h->n_dense = (int)dense.size();
        h->dense_floats = goff.back();
        h->dense_rows = roff.back();
        if (h->n_dense > 0) {
            // rows per CTA: 128-row tiles whose two accumulators (dim
            // columns each) fit the 512 tensor-memory columns, at most four
            const int mt = dense_mtiles(h->dense_max_dim);
            h->dense_groups = (h->dense_max_rows + mt * 128 - 1) / (mt * 128);
        }
        dense_off = goff;
        dense_off.insert(dense_off.end(), roff.begin(), roff.end());
    }
    std::vector<int32_t> order;
    {
        std::vector<std::vector<int32_t>> by_class(kNumClasses);
        for (int t = 0; t < num_tables; ++t) {
            h->tabs[t].cls = backward_class(h->tabs[t], h->total_d);
            if (h->tabs[t].dslot < 0) by_class[h->tabs[t].cls].push_back(t);
        }
        for (int c = 0; c < kNumClasses; ++c) {
            h->class_begin[c] = (int)order.size();
            h->class_count[c] = (int)by_class[c].size();
            order.insert(order.end(), by_class[c].begin(), by_class[c].end());
        }
    }
    const size_t bytes = dev_block_bytes(num_tables);
    e = cudaMalloc(&h->dev, bytes);
    if (e != cudaSuccess) {
        delete h;
        return e == cudaErrorMemoryAllocation ? TBE_ERR_NO_MEMORY : cuda_fail(e);
    }
    h->blk = static_cast<DevBlock*>(h->dev);
    h->dtabs = reinterpret_cast<TableDesc*>(static_cast<char*>(h->dev) + tabs_offset());
    h->dclass_tables = reinterpret_cast<int32_t*>(static_cast<char*>(h->dev) + class_list_offset(num_tables));
    h->dhist_tables = reinterpret_cast<int32_t*>(static_cast<char*>(h->dev) + hist_list_offset(num_tables));
    h->hist_f16.tables = h->dhist_tables;
    h->hist_bf16.tables = h->dhist_tables + hist_f16.size();
    h->ddense_tables = reinterpret_cast<int32_t*>(static_cast<char*>(h->dev) + dense_list_offset(num_tables));
    h->ddense_goff = reinterpret_cast<int64_t*>(static_cast<char*>(h->dev) + dense_off_offset(num_tables));
    h->ddense_roff = h->ddense_goff + (h->n_dense + 1);
    e = cudaMemset(h->dev, 0, tabs_offset());
    if (e == cudaSuccess)
        e = cudaMemcpy(h->dtabs, h->tabs.data(), sizeof(TableDesc) * num_tables, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !order.empty())  // dense tables are in no class list
        e = cudaMemcpy(h->dclass_tables, order.data(), sizeof(int32_t) * order.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !hist_f16.empty())
        e = cudaMemcpy(h->dhist_tables, hist_f16.data(), sizeof(int32_t) * hist_f16.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !hist_bf16.empty())
        e = cudaMemcpy(h->dhist_tables + hist_f16.size(), hist_bf16.data(), sizeof(int32_t) * hist_bf16.size(),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !dense.empty())
        e = cudaMemcpy(h->ddense_tables, dense.data(), sizeof(int32_t) * dense.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(h->ddense_goff, dense_off.data(), sizeof(int64_t) * dense_off.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(h->dev);
        delete h;
        return cuda_fail(e);
    }
    {
        int least = 0, greatest = 0;
        e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, greatest);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_apply_fork, cudaEventDisableTiming);
        for (int i = 0; i < kApplyStreams && e == cudaSuccess; ++i) {
            e = cudaStreamCreateWithFlags(&h->apply_streams[i], cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_apply_join[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            tbe_destroy(h);
            return cuda_fail(e);
        }
    }
    *out = h;
    return TBE_OK;
}

void tbe_destroy(tbe_handle* h) {
    if (!h) return;
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->side) cudaStreamDestroy(h->side);
    if (h->ev_apply_fork) cudaEventDestroy(h->ev_apply_fork);
    for (int i = 0; i < kApplyStreams; ++i) {
        if (h->ev_apply_join[i]) cudaEventDestroy(h->ev_apply_join[i]);
        if (h->apply_streams[i]) cudaStreamDestroy(h->apply_streams[i]);
    }
    if (h->dev) cudaFree(h->dev);
    if (h->dorder) cudaFree(h->dorder);
    delete h;
}

int tbe_forward(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                int64_t num_indices, int32_t batch_size, const float* per_sample_weights, float* out,
                void* stream) {
    CallRange range("tbe_forward");
    int rc = check_batch(h, indices, offsets, index_dtype, num_indices, batch_size);
    if (rc) return rc;
    if (batch_size == 0) return TBE_OK;
    if (!out) return TBE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = ensure_schedule(h, batch_size, s);
    if (rc) return rc;
    int64_t warps = 0;
    for (const TableDesc& d : h->tabs) {
        if (d.path == PATH_HIST) continue;
        const int per = d.path == PATH_VEC ? 32 / d.lanes : 1;
        const int blocks = d.path == PATH_VEC ? d.vecs : 1;
        warps += (int64_t)(batch_size + per - 1) / per * blocks;
    }
    if (warps >= (int64_t(1) << 31) / 32) return TBE_ERR_UNSUPPORTED;
    FwdArgs a{};
    a.tabs = h->dtabs;
    a.blk = h->blk;
    a.T = h->T;
    a.B = batch_size;
    a.N = num_indices;
    a.indices = indices;
    a.offsets = offsets;
    a.idx64 = index_dtype == TBE_I64;
    a.weights = per_sample_weights;
    a.mean = h->pooling == TBE_POOL_MEAN;
    a.out = out;
    a.total_d = h->total_d;
    a.vec_out = h->vec_out && ((uintptr_t)out % 16 == 0);
    a.total_warps = (int)warps;
    a.parity = h->parity;
    a.num_sms = h->num_sms;
    if (h->dorder) {  // TBE_FLAG_LENGTH_ORDER
        a.lcount = static_cast<uint32_t*>(h->dorder);
        a.lflag = a.lcount + (size_t)h->T * kLenBuckets;
        a.ldone = a.lflag + h->T;
        a.order = a.ldone + h->T;
    }
    rc = cuda_status(launch_forward(a, s));
    if (rc == TBE_OK && h->hist_f16.n + h->hist_bf16.n > 0)
        rc = cuda_status(launch_hist(a, h->hist_f16, h->hist_bf16, s));
    if (rc == TBE_OK) h->parity ^= 1;
    return rc;
}

int tbe_per_sample_weight_grad(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                               int64_t num_indices, int32_t batch_size, const float* grad_out,
                               float* grad_weights, void* stream) {
    CallRange range("tbe_per_sample_weight_grad");
    int rc = check_batch(h, indices, offsets, index_dtype, num_indices, batch_size);
    if (rc) return rc;
    if (batch_size == 0 || num_indices == 0) return TBE_OK;
    if (!grad_out || !grad_weights) return TBE_ERR_INVALID_ARG;
    if ((int64_t)h->T * batch_size >= (int64_t(1) << 31) / 32) return TBE_ERR_UNSUPPORTED;
    WgradArgs a{};
    a.tabs = h->dtabs;
    a.blk = h->blk;
    a.T = h->T;
    a.B = batch_size;
    a.N = num_indices;
    a.indices = indices;
    a.offsets = offsets;
    a.idx64 = index_dtype == TBE_I64;
    a.grad = grad_out;
    a.total_d = h->total_d;
    a.grad_vec = h->total_d % 4 == 0 && ((uintptr_t)grad_out % 16) == 0;
    a.mean = h->pooling == TBE_POOL_MEAN;
    a.out = grad_weights;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->flags & TBE_FLAG_LENGTH_ORDER) {
        // the forward's length-keyed bag order, computed for this batch
        rc = ensure_order(h, batch_size);
        if (rc) return rc;
        FwdArgs o{};
        o.tabs = h->dtabs;
        o.T = h->T;
        o.B = batch_size;
        o.offsets = offsets;
        o.idx64 = a.idx64;
        o.lcount = static_cast<uint32_t*>(h->dorder);
        o.lflag = o.lcount + (size_t)h->T * kLenBuckets;
        o.ldone = o.lflag + h->T;
        o.order = o.ldone + h->T;
        rc = cuda_status(launch_bag_order(o, s));
        if (rc) return rc;
        a.lflag = o.lflag;
        a.order = o.order;
    }
    return cuda_status(launch_wgrad(a, s));
}

size_t tbe_backward_workspace_bytes(const tbe_handle* h, int64_t num_indices, int32_t batch_size) {
    (void)batch_size;
    if (!h || num_indices < 0) return 0;
    return make_layout(h, num_indices, batch_size, kLayoutWithScale).total;
}

int tbe_backward_workspace_layout(const tbe_handle* h, int64_t num_indices, int32_t batch_size,
                                  tbe_ws_layout* out) {
    (void)batch_size;
    if (!h || !out || num_indices < 0) return TBE_ERR_INVALID_ARG;
    const Layout L = make_layout(h, num_indices, batch_size, kLayoutWithScale);
    const bool odd = h->passes % 2 == 1;
    out->sorted_keys = odd ? L.keys1 : L.keys0;
    out->sorted_vals = odd ? L.vals1 : L.vals0;
    out->uniq = L.uniq;
    out->runstart = L.runstart;
    out->num_unique = L.counters + sizeof(uint32_t) * CTR_U;
    out->total_bytes = L.total;
    return TBE_OK;
}

int tbe_backward_prepare(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                         int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                         void* workspace, size_t workspace_bytes, void* stream) {
    CallRange range("tbe_backward_prepare");
    int rc = check_batch(h, indices, offsets, index_dtype, num_indices, batch_size);
    if (rc) return rc;
    if (!workspace) return TBE_ERR_INVALID_ARG;
    const Layout L = make_layout(h, num_indices, batch_size, kLayoutWithScale);
    if (workspace_bytes < L.total) return TBE_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool scale = needs_scale(h, per_sample_weights);
    Workspace w = bind(h, L, workspace, scale);
    cudaError_t e = cudaMemsetAsync(workspace, 0, L.zero_bytes, s);
    if (e == cudaSuccess && num_indices == 0) e = cudaMemsetAsync(w.runstart, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
    // remember, in the workspace's counter block, whether a scale array was written
    if (scale) e = cudaMemsetAsync(w.counters + CTR_HAS_SCALE, 0xff, sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
    PrepArgs a{};
    a.tabs = h->dtabs;
    a.blk = h->blk;
    a.T = h->T;
    a.B = batch_size;
    a.N = num_indices;
    a.indices = indices;
    a.offsets = offsets;
    a.idx64 = index_dtype == TBE_I64;
    a.weights = per_sample_weights;
    a.mean = h->pooling == TBE_POOL_MEAN;
    a.total_rows = (uint32_t)h->total_rows;
    a.key_bits = h->key_bits;
    a.digit_bits = h->digit_bits;
    a.compact = h->n_dense > 0;
    a.chunk = long_chunk_lookups(num_indices, h->num_sms);
    return cuda_status(launch_prepare(a, w, s));
}

int tbe_forward_prepare(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                        int64_t num_indices, int32_t batch_size, const float* per_sample_weights, float* out,
                        void* workspace, size_t workspace_bytes, void* stream) {
    CallRange range("tbe_forward_prepare");
    int rc = check_batch(h, indices, offsets, index_dtype, num_indices, batch_size);
    if (rc) return rc;
    if (!workspace || (batch_size > 0 && !out)) return TBE_ERR_INVALID_ARG;
    if (workspace_bytes < make_layout(h, num_indices, batch_size, kLayoutWithScale).total) return TBE_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // fork: the side stream starts after everything already queued on s
    cudaError_t fe = cudaEventRecord(h->ev_fork, s);
    if (fe == cudaSuccess) fe = cudaStreamWaitEvent(h->side, h->ev_fork, 0);
    if (fe != cudaSuccess) return cuda_fail(fe);
    rc = tbe_backward_prepare(h, indices, offsets, index_dtype, num_indices, batch_size, per_sample_weights,
                              workspace, workspace_bytes, h->side);
    // the forward pass runs on s meanwhile
    if (rc == TBE_OK)
        rc = tbe_forward(h, indices, offsets, index_dtype, num_indices, batch_size, per_sample_weights, out, stream);
    // join: later work on s waits for the preparation (also after an error,
    // so s never runs ahead of work already queued on the side stream)
    const bool joined = cudaEventRecord(h->ev_join, h->side) == cudaSuccess &&
                        cudaStreamWaitEvent(s, h->ev_join, 0) == cudaSuccess;
    if (rc) return rc;
    return joined ? TBE_OK : TBE_ERR_CUDA;
}

int tbe_backward_apply(tbe_handle* h, int64_t num_indices, int32_t batch_size, const float* grad_out,
                       const tbe_optimizer* opt, void* workspace, size_t workspace_bytes, void* stream) {
    CallRange range("tbe_backward_apply");
    if (!h || !opt || !workspace) return TBE_ERR_INVALID_ARG;
    if (!on_handle_device(h)) return TBE_ERR_INVALID_ARG;
    if (num_indices < 0 || batch_size < 0) return TBE_ERR_INVALID_ARG;
    if (num_indices >= (int64_t(1) << 30)) return TBE_ERR_UNSUPPORTED;
    if (opt->kind != TBE_OPT_SGD && opt->kind != TBE_OPT_ROWWISE_ADAGRAD) return TBE_ERR_INVALID_ARG;
    if (opt->kind == TBE_OPT_ROWWISE_ADAGRAD && !opt->state) return TBE_ERR_INVALID_ARG;
    if (num_indices > 0 && !grad_out) return TBE_ERR_INVALID_ARG;
    const Layout L = make_layout(h, num_indices, batch_size, kLayoutWithScale);
    if (workspace_bytes < L.total) return TBE_ERR_WORKSPACE_TOO_SMALL;
    if (num_indices == 0 || batch_size == 0) return TBE_OK;
    Workspace w = bind(h, L, workspace, true);
    ApplyArgs a{};
    a.tabs = h->dtabs;
    a.blk = h->blk;
    a.T = h->T;
    a.B = batch_size;
    a.N = num_indices;
    a.grad = grad_out;
    a.grad_vec = ((uintptr_t)grad_out % 16) == 0;
    a.total_d = h->total_d;
    a.part_stride = part_stride(h);
    a.chunk = long_chunk_lookups(num_indices, h->num_sms);
    a.total_rows = (uint32_t)h->total_rows;
    a.has_scale = 0;
    a.opt = opt->kind;
    a.lr = opt->lr;
    a.eps = opt->eps;
    a.state = opt->state;
    a.num_sms = h->num_sms;
    DenseArgs d{};
    d.tabs = h->dtabs;
    d.blk = h->blk;
    d.B = batch_size;
    d.grad = grad_out;
    d.total_d = h->total_d;
    d.opt = opt->kind;
    d.lr = opt->lr;
    d.eps = opt->eps;
    d.state = opt->state;
    d.tables = h->ddense_tables;
    d.goff = h->ddense_goff;
    d.roff = h->ddense_roff;
    d.n = h->n_dense;
    d.max_rows = h->dense_max_rows;
    d.max_dim = h->dense_max_dim;
    d.num_sms = h->num_sms;
    d.total_rows = h->dense_rows;
    d.total_floats = h->dense_floats;
    d.splits = dense_parts(h, batch_size);
    d.grad_vec = ((uintptr_t)grad_out % 16) == 0 && h->total_d % 4 == 0;
    return cuda_status(launch_apply(a, w, h->dclass_tables, h->class_begin, h->class_count,
                                    h->n_dense > 0 ? &d : nullptr,
                                    static_cast<cudaStream_t>(stream), h->apply_streams, h->ev_apply_fork,
                                    h->ev_apply_join));
}

int tbe_backward_sgd(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                     int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                     const float* grad_out, float lr, void* workspace, size_t workspace_bytes,
                     void* stream) {
    CallRange range("tbe_backward_sgd");
    int rc = tbe_backward_prepare(h, indices, offsets, index_dtype, num_indices, batch_size,
                                  per_sample_weights, workspace, workspace_bytes, stream);
    if (rc) return rc;
    tbe_optimizer o{TBE_OPT_SGD, lr, 0.f, nullptr};
    return tbe_backward_apply(h, num_indices, batch_size, grad_out, &o, workspace, workspace_bytes, stream);
}

int tbe_backward_rowwise_adagrad(tbe_handle* h, const void* indices, const void* offsets,
                                 int32_t index_dtype, int64_t num_indices, int32_t batch_size,
                                 const float* per_sample_weights, const float* grad_out, float* state,
                                 float lr, float eps, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    CallRange range("tbe_backward_rowwise_adagrad");
    if (!state) return TBE_ERR_INVALID_ARG;
    int rc = tbe_backward_prepare(h, indices, offsets, index_dtype, num_indices, batch_size,
                                  per_sample_weights, workspace, workspace_bytes, stream);
    if (rc) return rc;
    tbe_optimizer o{TBE_OPT_ROWWISE_ADAGRAD, lr, eps, state};
    return tbe_backward_apply(h, num_indices, batch_size, grad_out, &o, workspace, workspace_bytes, stream);
}

int tbe_get_error(tbe_handle* h, void* stream) {
    if (!h || !on_handle_device(h)) return TBE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    cudaError_t e = cudaMemcpyAsync(&bits, &h->blk->error, sizeof bits, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&h->blk->error, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (bits & ERR_TIMEOUT) return TBE_ERR_TIMEOUT;
    if (bits & ERR_OFFSETS) return TBE_ERR_BAD_OFFSETS;
    if (bits & ERR_OOB) return TBE_ERR_INDEX_OOB;
    return TBE_OK;
}

int tbe_last_cuda_error(void) { return (int)g_last_cuda_error; }

const char* tbe_strerror(int code) {
    switch (code) {
        case TBE_OK: return "ok";
        case TBE_ERR_INVALID_ARG: return "invalid argument";
        case TBE_ERR_UNSUPPORTED: return "unsupported size or layout";
        case TBE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case TBE_ERR_CUDA: return "CUDA runtime error";
        case TBE_ERR_INDEX_OOB: return "index out of range (lookup skipped)";
        case TBE_ERR_BAD_OFFSETS: return "offsets not monotone from 0 to N";
        case TBE_ERR_TIMEOUT: return "bounded device wait ran out";
        case TBE_ERR_NO_MEMORY: return "out of memory";
        default: return "unknown error";
    }
}

int tbe_table_paths(const tbe_handle* h, int32_t* out_path) {
    if (!h || !out_path) return TBE_ERR_INVALID_ARG;
    for (int t = 0; t < h->T; ++t) out_path[t] = h->tabs[t].path;
    return TBE_OK;
}

int tbe_table_backward_paths(const tbe_handle* h, int32_t* out_path) {
    if (!h || !out_path) return TBE_ERR_INVALID_ARG;
    for (int t = 0; t < h->T; ++t) out_path[t] = h->tabs[t].dslot >= 0 ? 1 : 0;
    return TBE_OK;
}

}  // extern "C"
