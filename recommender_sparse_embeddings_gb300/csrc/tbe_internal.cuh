// Internal definitions shared by the TBE kernels and the C ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tbe {

enum : int32_t { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

// Sticky device error bits (one word in the descriptor block).
enum : uint32_t { ERR_OOB = 1u, ERR_OFFSETS = 2u, ERR_TIMEOUT = 4u };

// Forward gather schedule of one table.
enum : int32_t { PATH_VEC = 0, PATH_SCALAR = 1, PATH_HIST = 2 };

// Most tables one handle may hold.
constexpr int kMaxTables = 4096;
// Bags longer than this are pooled by a whole CTA instead of one slot.
constexpr int kLongBag = 2048;
// Capacity of the long-bag list held in the descriptor block.
constexpr int kLongBagCap = 1 << 16;
// Runs of at least this many lookups take the chunked accumulate path.
constexpr int kLongRun = 256;
// Lookups per chunk of a long run for a batch of N lookups: 256, doubled up
// to 1024 while the batch still makes at least eight chunks per apply warp
// (3 CTAs of 8 warps per SM), so big batches take fewer, longer work items.
inline int long_chunk_lookups(int64_t N, int num_sms) {
    const int64_t warps = (int64_t)num_sms * 3 * 8;
    int c = kLongRun;
    while (c < 4 * kLongRun && N / (2 * c) >= 8 * warps) c *= 2;
    return c;
}
// Keys per tile of the key, sort and run-length kernels (256 threads x 16).
constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;
// Radix digits are 8 bits, or 9 when that saves a pass (keys of 17-18 or
// 25-27 bits); arrays are sized for the larger.
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kMaxRadixBits = 9;
constexpr int kMaxRadix = 1 << kMaxRadixBits;
constexpr int kMaxPasses = 4;
// Iteration limit of every spin wait (each iteration sleeps ~64 ns).
constexpr int kSpinLimit = 1 << 20;

struct TableDesc {
    void* data;       // device, row-major rows x dim
    int64_t rows;
    int64_t rowbase;  // sum of rows of the tables before this one
    int32_t dim;
    int32_t doff;       // first output column
    int32_t dtype;      // DT_*
    int32_t row_bytes;  // dim * element size
    int32_t path;       // PATH_*
    int32_t lanes;      // lanes per row slice in the vector path (power of 2, <= 32)
    int32_t vecs;       // column blocks of 32 vectors per row (vector path, 1..4)
    int32_t warp_begin; // first warp of this table in the forward warp map
    int32_t cls;        // backward class: dtype * NUM_SHAPES + row shape code
    int32_t dslot;      // index among the dense-backward tables, -1 for the sorted path
};

// Device-resident descriptor block owned by a handle.
struct DevBlock {
    uint32_t error;        // sticky ERR_* bits
    uint32_t long_count[2];// long-bag list fill counters (alternate per call)
    uint32_t pad;
    uint64_t long_bags[2][kLongBagCap];  // flat bag ids of bags longer than kLongBag
    // TableDesc tables[T] follows (aligned to 64 bytes)
};

__host__ __device__ inline int elem_bytes(int dt) { return dt == DT_F32 ? 4 : 2; }

template <typename T>
__host__ __device__ __forceinline__ T tmin(T a, T b) { return b < a ? b : a; }
template <typename T>
__host__ __device__ __forceinline__ T tmax(T a, T b) { return a < b ? b : a; }

// ------------------------------------------------------------ conversions

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ float h_bits_to_float(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)h));
}

// Element k of a row as float.
template <int DT>
__device__ __forceinline__ float load_elem(const void* base, int64_t k) {
    if constexpr (DT == DT_F32) {
        return __ldg(reinterpret_cast<const float*>(base) + k);
    } else if constexpr (DT == DT_F16) {
        return __half2float(__ldg(reinterpret_cast<const __half*>(base) + k));
    } else {
        return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + k));
    }
}

template <int DT>
__device__ __forceinline__ void store_elem(void* base, int64_t k, float v) {
    if constexpr (DT == DT_F32) {
        reinterpret_cast<float*>(base)[k] = v;
    } else if constexpr (DT == DT_F16) {
        reinterpret_cast<__half*>(base)[k] = __float2half_rn(v);
    } else {
        reinterpret_cast<__nv_bfloat16*>(base)[k] = __float2bfloat16_rn(v);
    }
}

// acc += s * (x, y) on both halves of a float pair, one packed fp32 FMA
// (each half rounds exactly like fmaf).
__device__ __forceinline__ void ffma2(float& a0, float& a1, float s, float x, float y) {
    asm("{\n\t.reg .b64 p, q, r;\n\t"
        "mov.b64 p, {%2, %2};\n\t"
        "mov.b64 q, {%3, %4};\n\t"
        "mov.b64 r, {%0, %1};\n\t"
        "fma.rn.f32x2 r, p, q, r;\n\t"
        "mov.b64 {%0, %1}, r;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s), "f"(x), "f"(y));
}

// Compensated (Kahan) addition of (x0, x1) into the sums (s0, s1) with
// compensations (c0, c1), both halves at once with packed fp32 adds (each
// half rounds exactly like the scalar steps y = x - c, t = s + y,
// c = (t - s) - y, s = t).
__device__ __forceinline__ void kahan2(float& s0, float& s1, float& c0, float& c1, float x0, float x1) {
    asm("{\n\t.reg .b64 S, C, X, Y, T, D;\n\t"
        "mov.b64 S, {%0, %1};\n\t"
        "mov.b64 C, {%2, %3};\n\t"
        "mov.b64 X, {%4, %5};\n\t"
        "sub.rn.f32x2 Y, X, C;\n\t"
        "add.rn.f32x2 T, S, Y;\n\t"
        "sub.rn.f32x2 D, T, S;\n\t"
        "sub.rn.f32x2 C, D, Y;\n\t"
        "mov.b64 {%0, %1}, T;\n\t"
        "mov.b64 {%2, %3}, C;\n\t}"
        : "+f"(s0), "+f"(s1), "+f"(c0), "+f"(c1)
        : "f"(x0), "f"(x1));
}

// Unpack one 16-byte vector of DT into E = 16/sizeof(DT) floats.
template <int DT>
__device__ __forceinline__ void unpack16(const uint4& v, float* f) {
    if constexpr (DT == DT_F32) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (DT == DT_F16) {
                f[2 * i] = h_bits_to_float(w[i] & 0xffffu);
                f[2 * i + 1] = h_bits_to_float(w[i] >> 16);
            } else {
                f[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
                f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
            }
        }
    }
}

// Chained launches (programmatic dependent launch).  A kernel started with
// launch_chained may be launched before the kernel ahead of it on the stream
// has completed: once every CTA of that kernel has exited, its CTAs are
// placed at once instead of after the grid's completion is processed.  Its
// first statement, chain_wait(), waits until that kernel has completed and
// its writes are visible, so every kernel launched this way keeps the order
// of the stream.  No kernel releases its dependents early: CTAs waiting on
// an SM would hold resources that a kernel on another stream could use.
__device__ __forceinline__ void chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args... args) {
    return launch_chained_smem(kernel, grid, block, 0, s, args...);
}

template <typename IDX>
__device__ __forceinline__ int64_t ld_index(const IDX* p, int64_t k) {
    return (int64_t)__ldg(p + k);
}

// ------------------------------------------------------------ launch API
// (host functions defined in the kernel files, called by the ABI layer)

struct FwdArgs {
    const TableDesc* tabs;
    DevBlock* blk;
    int T;
    int B;
    int64_t N;
    const void* indices;
    const void* offsets;
    int idx64;
    const float* weights;
    int mean;
    float* out;
    int total_d;
    int vec_out;   // output rows and column offsets allow 16-byte stores
    int total_warps;
    int parity;    // which long-bag counter this call uses
    int num_sms;
    // length-keyed bag order (null: bags in index order): per table, the
    // count of its bags of each length bucket (then the buckets' starts),
    // whether its bags differ in length, and its bags ordered by length
    uint32_t* lcount;  // [T][kLenBuckets]
    uint32_t* lflag;   // [T]
    uint32_t* ldone;   // [T]: CTAs of the table done (zero between calls)
    uint32_t* order;   // [T][B]
};

// Bag-length buckets of the length-keyed order: lengths 0 .. kLenBuckets-2,
// and longer ones together.
constexpr int kLenBuckets = 256;

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s);
// The length-keyed bag order alone (reads T, B, offsets, idx64, tabs and
// the order arrays of a).
cudaError_t launch_bag_order(const FwdArgs& a, cudaStream_t s);

// Gradient of the per-sample weights (wgrad.cu).
struct WgradArgs {
    const TableDesc* tabs;
    DevBlock* blk;
    int T;
    int B;
    int64_t N;
    const void* indices;
    const void* offsets;
    int idx64;
    const float* grad;  // [B, total_d]
    int total_d;
    int grad_vec;       // grad rows and table column offsets allow 16-byte loads
    int mean;
    float* out;         // [N]
    // length-keyed bag order (null: index order), as the forward's
    const uint32_t* lflag;  // [T]
    const uint32_t* order;  // [T][B]
};

// With a.order set, the bag order was just launched on s and the kernel
// follows it chained.
cudaError_t launch_wgrad(const WgradArgs& a, cudaStream_t s);

// Small-table tensor-core path (hist.cu).  One launch per table dtype.
struct HistGroup {
    const int32_t* tables;  // device: the group's tables
    int n;
    int dmax;         // largest dim
    int kmax;         // largest row count padded to 64
    size_t wt_bytes;  // largest dim x padded rows x 2 (one table's W^T)
    size_t smem;      // dynamic shared memory of the launch
};
size_t hist_smem_bytes(int kmax, size_t wt_bytes);
cudaError_t hist_configure(int optin_smem);
cudaError_t launch_hist(const FwdArgs& a, const HistGroup& f16, const HistGroup& bf16, cudaStream_t s);

struct Workspace {
    uint32_t* counters;   // [64]
    uint32_t* hist;       // [kMaxPasses][kMaxRadix]
    uint32_t* tcount;     // [1 << digit_bits][tiles]: digit counts of each tile, then digit starts
    uint32_t* tile_bag;   // [tiles]: first bag of each key tile (zeroed per call)
    uint32_t* keys[2];    // [N] ping-pong
    uint32_t* vals[2];    // [N] ping-pong: with scale, each lookup's position; without, its flat bag
    uint32_t* bag;        // [N] flat bag of each position (written only with scale)
    float* scale;         // [N] s_i of each position (weights and/or mean)
    uint32_t* uniq;       // [N]
    uint32_t* runstart;   // [N+1]
    uint2* chunk_info;    // [max_chunks]: (distinct-key index u of the run, first chunk of the run)
    uint32_t* chunk_done; // [max_chunks]: chunks of the run finished, kept at the run's first chunk
    uint32_t* cstart;     // [T+1]: first chunk of each table's long runs (cstart[T]: total)
    uint32_t* ustart;     // [T+1]: first distinct-key index of each table (ustart[T]: end)
    uint32_t* tpos;       // [T+1]: position of each table's first lookup (tpos[T] = N)
    uint32_t* cbase;      // [T+1]: first sorted slot of each sorted-path table's keys (compacted)
    uint16_t* hrow;       // [N]: row of each dense-table lookup (0xffff: skipped)
    uint32_t* dboff;      // [dense tables][B+1]: offsets of each dense table's bags
    float* dgrad;         // [splits][dense floats]: dense tables' partial gradients, row-major per table
    uint32_t* dcount;     // dense tables' lookups per row
    int compact;          // dense tables present: their lookups stay out of the sort
    float* partial;       // [max_chunks][part_stride]
    int64_t max_chunks;
    int tiles;
    int passes;
    int digit_bits;       // 8 or 9
    int sorted_buf;       // which ping-pong buffer holds the sorted result
};

// Counter slots inside Workspace::counters.
enum : int {
    CTR_U = 0,          // number of distinct keys
    CTR_NS = 1,         // number of sorted keys (lookups of sorted-path tables)
    CTR_NCHUNK = 2,     // number of chunks of long runs
    CTR_WORK = 8,       // apply work-item counters, one per backward class [15]
    CTR_EXIT = 24,      // apply finished-warp counters, one per backward class [15]
    CTR_HAS_SCALE = 63, // nonzero when prepare wrote the per-lookup scale array
    CTR_COUNT = 64,
};

struct PrepArgs {
    const TableDesc* tabs;
    DevBlock* blk;
    int T;
    int B;
    int64_t N;
    const void* indices;
    const void* offsets;
    int idx64;
    const float* weights;
    int mean;
    uint32_t total_rows;  // sentinel key for skipped lookups
    int key_bits;
    int digit_bits;  // radix digit width (8 or 9)
    int compact;     // dense tables present (their lookups are not sorted)
    int chunk;       // lookups per chunk of a long run (long_chunk_lookups)
};

// Backward row-shape codes: dim 32, 64, 128, 256 with aligned rows and
// gradient columns get vector lanes (VW columns per lane, NB blocks of 32*VW);
// every other table is element-wise (code 0).
enum : int { SHAPE_GENERIC = 0, SHAPE_D32 = 1, SHAPE_D64 = 2, SHAPE_D128 = 3, SHAPE_D256 = 4, NUM_SHAPES = 5 };
constexpr int kNumClasses = 3 * NUM_SHAPES;

cudaError_t launch_prepare(const PrepArgs& a, Workspace& ws, cudaStream_t s);

struct ApplyArgs {
    const TableDesc* tabs;
    DevBlock* blk;
    int T;
    int B;
    int64_t N;
    const float* grad;
    int grad_vec;  // grad is 16-byte aligned (vector loads allowed)
    int total_d;
    int part_stride;  // floats per partial-sum row (multiple of 4)
    int chunk;        // lookups per chunk of a long run (as the preparation used)
    uint32_t total_rows;
    int has_scale;  // filled in on the device from CTR_HAS_SCALE
    int opt;
    float lr;
    float eps;
    float* state;
    int num_sms;
    const int32_t* class_tables;  // tables of the launched class (device)
    int class_count;
    int cls;
};

// Dense backward of the histogram tables (dense.cu): per table, the row
// gradients are summed in shared memory straight from the lookups (no sort),
// then every row some lookup touched gets one optimizer step.
struct DenseArgs {
    const TableDesc* tabs;
    DevBlock* blk;
    int B;
    const float* grad;
    int total_d;
    int opt;
    float lr;
    float eps;
    float* state;
    const int32_t* tables;   // dense tables (device)
    const int64_t* goff;     // [n+1] first gradient float of each dense table in dgrad (device)
    const int64_t* roff;     // [n+1] first row count of each dense table in dcount (device)
    int n;
    int max_rows;
    int max_dim;
    int num_sms;
    int64_t total_rows;      // sum of the dense tables' rows (rows to update)
    int64_t total_floats;    // sum of the dense tables' rows x dims
    int splits;              // parts each table's bags are split into (one gradient slice each)
    int grad_vec;            // grad is 16-byte aligned with total_d % 4 == 0 (float4 rows)
};
cudaError_t dense_configure(int optin_smem);
cudaError_t launch_dense(const DenseArgs& a, const Workspace& ws, cudaStream_t s);

// 128-row M tiles per dense-backward CTA for dim D: the short and the long
// accumulator take D tensor-memory columns per tile each, 512 columns in all.
__host__ __device__ inline int dense_mtiles(int D) {
    const int by_tmem = 256 / D;
    return by_tmem < 4 ? (by_tmem < 1 ? 1 : by_tmem) : 4;
}

// Streams the backward class kernels are spread over: each class kernel
// takes its work from its own counter, so they may run side by side and one
// class's tail overlaps the next class's work.
constexpr int kApplyStreams = 4;

// One launch per backward class present: class_tables lists the tables of
// every class (device, grouped by class); class_begin/class_count index it.
// With more than one class, the launches fork from s onto the given streams
// and s waits for all.
// dense (nullable) runs side by side with the class kernels.
cudaError_t launch_apply(const ApplyArgs& a, const Workspace& ws, const int32_t* class_tables,
                         const int* class_begin, const int* class_count, const DenseArgs* dense,
                         cudaStream_t s, const cudaStream_t* streams, cudaEvent_t ev_fork,
                         const cudaEvent_t* ev_join);

}  // namespace tbe
