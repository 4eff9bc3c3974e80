// Host side of the C ABI declared in include/gdg.h: argument checks, TMA tensor-map
// encoding, form selection and kernel launches.  No device memory is allocated here and
// the host never waits on the GPU (except in gdg_device_error, which says so).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>

#include "gdg.h"
#include "grouped_gemm.cuh"

namespace {

using gdg::GemmParams;
using gdg::DenseParams;
using gdg::ReduceParams;

__device__ unsigned int g_device_error = 0;

constexpr int kMaxDevices = 64;

// ------------------------------------------------------------------ driver entry point

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map; OOB elements read as zero.
bool encode_map(CUtensorMap* m, CUtensorMapDataType type, CUtensorMapSwizzle swz,
                const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[4];
    cuuint64_t s[3];
    cuuint32_t b[4];
    cuuint32_t es[4] = {1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
    CUresult r = fn(m, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 operand map with 128-byte swizzle (the MMA's shared-memory layout).
bool encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
            const uint64_t* strides_bytes, const uint32_t* box) {
    return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, base, rank,
                      dims, strides_bytes, box);
}

// [rows, cols] bf16 as a plain 2-D map with box {64, box_rows}: one copy brings one 64-column
// block of box_rows rows (box_rows x 128 B); columns and rows past the extent read as zeros.
bool encode_rows_2d(CUtensorMap* m, const void* base, int64_t rows, int cols, uint32_t box_rows) {
    const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(cols) * 2};
    const uint32_t box[2] = {64, box_rows};
    return encode(m, base, 2, dims, strides, box);
}

// W [E, N, K] as {K, N, E} with box {64, 128, 1}: one copy brings 64 k-columns of 128 n-rows
// of one expert (a box never crosses into another expert; past N or K it reads zeros).
bool encode_weight_3d(CUtensorMap* m, const void* base, int E, int N, int K) {
    const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                              static_cast<uint64_t>(E)};
    const uint64_t strides[2] = {static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(N) * K * 2};
    const uint32_t box[3] = {64, 128, 1};
    return encode(m, base, 3, dims, strides, box);
}

// ------------------------------------------------------------------ per-device caches

struct DeviceInfo {
    std::atomic<int> ready{0};
    int sms = 0;
    int pairs = 0;              // co-resident CTA pairs of grouped_gemm_kernel
    unsigned int* err = nullptr;
    std::mutex mu;
};

DeviceInfo g_dev[kMaxDevices];

// Sets the kernel's shared-memory size and lowers *pairs to the number of CTA pairs of it
// that fit on the device at once (the persistent grid; every variant launches with the
// smallest).  The grid size never changes results, only speed.
template <int OP, int EPI, int RT>
cudaError_t set_up_kernel(int sms, int* pairs) {
    cudaError_t e = cudaFuncSetAttribute(gdg::grouped_gemm_kernel<OP, EPI, RT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gdg::kGemmSmemBytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(gdg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gdg::kGemmSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gdg::grouped_gemm_kernel<OP, EPI, RT>, &cfg) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        n = sms / 2;
    }
    if (n < *pairs) *pairs = n;
    return cudaSuccess;
}

// Per-device set-up, once: SM count, device error word address, kernel attributes.
DeviceInfo* device_info(gdg_status* st) {
    int dev = 0;
    // cudaSetDevice binds the device's primary context to this thread: the tensor-map encoder
    // is a driver-API call and needs a current context, which a thread that has made no
    // runtime call yet (an autograd worker thread, say) does not have.
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
        cudaSetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        *st = GDG_ECUDA;
        return nullptr;
    }
    DeviceInfo& d = g_dev[dev];
    if (d.ready.load(std::memory_order_acquire)) return &d;
    std::lock_guard<std::mutex> lock(d.mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
        void* err = nullptr;
        d.pairs = 1 << 20;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaGetSymbolAddress(&err, g_device_error) != cudaSuccess ||
            set_up_kernel<gdg::OP_FWD, gdg::EPI_BF16, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_FWD, gdg::EPI_BF16, 128>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_DGRAD, gdg::EPI_BF16, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_DGRAD, gdg::EPI_BF16, 128>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_WGRAD, gdg::EPI_BF16, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_WGRAD, gdg::EPI_FP32, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_WGRAD, gdg::EPI_BF16_ACC, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_WGRAD, gdg::EPI_FP32_ACC, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_WGRAD, gdg::EPI_PARTIAL, 256>(d.sms, &d.pairs) != cudaSuccess ||
            set_up_kernel<gdg::OP_WGRAD, gdg::EPI_RED, 256>(d.sms, &d.pairs) != cudaSuccess) {
            *st = GDG_ECUDA;
            return nullptr;
        }
        d.err = static_cast<unsigned int*>(err);
        d.ready.store(1, std::memory_order_release);
    }
    return &d;
}

// ------------------------------------------------------------------ checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void* p, uint64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The output's strides (elements) and the bytes it spans, from out_ld / out_es (0 = dense).
struct OutLayout {
    int64_t ld = 0, es = 0;
    uint64_t span = 0;
};

// out is [E][n][cols] with unit stride along cols (E = 1 and no expert stride for fwd / dgrad).
// Strides must keep every row on a 16-byte boundary (the epilogues store 16-byte chunks), and
// no two elements may share memory: taken in increasing order of stride, the row and expert
// strides must each reach past everything below them.
gdg_status out_layout(const gdg_args* a, int64_t n, int64_t cols, int64_t E, uint64_t esz,
                      bool wgrad, OutLayout* L) {
    if (a->out_ld < 0 || a->out_es < 0 || (!wgrad && a->out_es != 0)) return GDG_EINVAL;
    const int64_t ld = a->out_ld ? a->out_ld : cols;
    const int64_t es = !wgrad ? 0 : (a->out_es ? a->out_es : n * ld);
    if ((static_cast<uint64_t>(ld) * esz) % 16 != 0 || (static_cast<uint64_t>(es) * esz) % 16 != 0)
        return GDG_EALIGN;
    int64_t s1 = ld, n1 = n, s2 = es, n2 = E;       // (stride, extent) of the two outer dims
    if (n1 <= 1) { s1 = s2; n1 = n2; s2 = 0; n2 = 1; }
    if (n2 > 1 && s2 < s1) { std::swap(s1, s2); std::swap(n1, n2); }
    const int64_t below1 = cols;                     // span of the dims under the first
    if (n1 > 1 && s1 < below1) return GDG_EOVERLAP;
    const int64_t below2 = (n1 > 1 ? (n1 - 1) * s1 : 0) + cols;
    if (n2 > 1 && s2 < below2) return GDG_EOVERLAP;
    if (static_cast<double>(E - 1) * es + static_cast<double>(n - 1) * ld + cols > 9.0e15)
        return GDG_EINVAL;
    L->ld = ld;
    L->es = es;
    L->span = static_cast<uint64_t>((E - 1) * es + (n > 0 ? (n - 1) * ld : 0) + cols) * esz;
    return GDG_OK;
}

int tiles_per_expert(int N, int K) {
    return static_cast<int>(ceil_div(N, gdg::kPairM) * ceil_div(K, gdg::kBN));
}

// Persistent grid: two CTAs per pair, at most one pair per unit.
// Test-only cap on the pairs of a launch (0: none), set by gdg_test_set_max_pairs.
std::atomic<int> g_max_pairs{0};

int pair_grid(int64_t units, int pairs) {
    const int cap = g_max_pairs.load(std::memory_order_relaxed);
    if (cap > 0 && pairs > cap) pairs = cap;
    const int64_t n = units < pairs ? units : pairs;
    return static_cast<int>(2 * (n > 0 ? n : 1));
}

// wgrad, groups walked by size: the team schedule (grouped_gemm.cuh, assign_teams) when a
// group's tiles are fewer than the launch's pairs and at most kMaxTeams teams result.
int teams_rule(int sorted, int tiles_per_expert, int pairs) {
    if (!sorted || tiles_per_expert >= pairs) return 0;
    const int full = pairs / tiles_per_expert;
    const int nteams = full + (pairs % tiles_per_expert ? 1 : 0);
    return nteams <= gdg::kMaxTeams ? 1 : 0;
}

// wgrad, unsplit: walk the groups by decreasing size when groups are long on average (at least
// 512 rows): the tiles of one group then run side by side and its rows come from HBM once.
// A rule on shapes only.
int sort_groups_rule(int64_t rows, int E) {
    return (E <= gdg::kMaxSorted && rows >= static_cast<int64_t>(E) * 512) ? 1 : 0;
}

int32_t auto_split_rows(int64_t rows, int E, int N, int K) {
    const int64_t tpe = tiles_per_expert(N, K);
    // Shapes with few output tiles leave SMs idle in the unsplit form; cut the rows of
    // each group into fixed chunks instead, when the groups are long enough (6144 rows on
    // average) for the shorter units to repay the ordered reduce: measured, 8192-row groups
    // gain 17 % (E = 2, N = K = 1024) and 4096-row groups lose 6-14 % (E = 8, N = K = 512).
    // The rule looks at shapes only, so the bits never depend on the GPU it runs on.
    if (rows <= 0 || static_cast<int64_t>(E) * tpe >= 64 || rows < static_cast<int64_t>(E) * 6144)
        return -1;
    int64_t r = ceil_div(rows * tpe, 128);
    r = ceil_div(r, 64) * 64;
    if (r < 128) r = 128;
    if (r > (1 << 30)) r = 1 << 30;
    return static_cast<int32_t>(r);
}

int64_t split_max_units(int64_t rows, int E, int N, int K, int32_t split_rows) {
    return static_cast<int64_t>(tiles_per_expert(N, K)) * (ceil_div(rows, split_rows) + E);
}

gdg_status check_common(const gdg_args* args, const int32_t* offs, int E, int N, int K,
                        gdg_dtype out_dtype) {
    if (!args) return GDG_EINVAL;
    if (E < 1 || E > GDG_MAX_EXPERTS || N <= 0 || K <= 0 || args->rows < 0 ||
        args->rows > GDG_MAX_ROWS)
        return GDG_EINVAL;
    if (args->offs_kind != GDG_OFFS_ENDS && args->offs_kind != GDG_OFFS_INDPTR) return GDG_EINVAL;
    if (out_dtype != GDG_BF16 && out_dtype != GDG_FP32) return GDG_EINVAL;
    if (N % 8 != 0 || K % 8 != 0) return GDG_EALIGN;   // 16-byte rows: TMA strides
    if (static_cast<int64_t>(E) * N * K > (int64_t{1} << 40)) return GDG_EINVAL;
    if (static_cast<int64_t>(E) * N >= INT32_MAX) return GDG_EINVAL;   // TMA row coordinates
    if (!offs) return GDG_EINVAL;
    (void)offs;
    return GDG_OK;
}

gdg_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return GDG_OK;
    cudaGetLastError();   // clear a sticky launch-config error so later calls can proceed
    return GDG_ECUDA;
}

// A validated call with everything its launches need, bound once: the kernel variant, the
// encoded tensor maps and parameters, and the grid.  Launching it does no host work beyond
// the kernel launches, allocates nothing and never synchronises.
struct Plan {
    int op = 0;              // GDG_OP_*
    int rt = 256;            // fwd / dgrad row tile (ring geometry)
    int epi = 0;             // wgrad kernel's epilogue (EPI_PARTIAL for the split form)
    bool launch = false;     // false: the call has nothing to launch (rows == 0 cases)
    bool reduce = false;     // split form: ordered reduce of the partials after the GEMM
    bool zero = false;       // unordered split form: zero the fp32 destination first
    bool finish = false;     // unordered split form, bf16 out: round the fp32 sums into out
    int grid = 0;
    int rgrid = 0;
    GemmParams p;
    ReduceParams r;
    DenseParams z;           // zero kernel
    DenseParams f;           // finish kernel
};

// fwd (OP_FWD) and dgrad (OP_DGRAD) share everything but the operand maps.
template <int OP>
gdg_status plan_fwd_like(const gdg_args* args, const int32_t* offs, int E, int N, int K,
                         gdg_dtype out_dtype, int accumulate, Plan* pl) {
    gdg_status st = check_common(args, offs, E, N, K, out_dtype);
    if (st != GDG_OK) return st;
    if (out_dtype != GDG_BF16 || accumulate != 0 || args->split_rows != 0) return GDG_EINVAL;
    const int64_t rows = args->rows;
    pl->op = OP;
    pl->launch = false;
    if (rows == 0) return GDG_OK;
    if (!args->a || !args->b || !args->out) return GDG_EINVAL;
    if (!aligned16(args->a) || !aligned16(args->b) || !aligned16(args->out) || !aligned16(offs))
        return GDG_EALIGN;
    const int in_cols = (OP == gdg::OP_FWD) ? K : N;     // columns of the row operand
    const int out_cols = (OP == gdg::OP_FWD) ? N : K;
    OutLayout L;
    st = out_layout(args, rows, out_cols, 1, 2, false, &L);
    if (st != GDG_OK) return st;
    const Range r_out = range_of(args->out, L.span);
    const Range r_a = range_of(args->a, static_cast<uint64_t>(rows) * in_cols * 2);
    const Range r_b = range_of(args->b, static_cast<uint64_t>(E) * N * K * 2);
    const Range r_o = range_of(offs, static_cast<uint64_t>(E + args->offs_kind) * 4);
    if (overlaps(r_out, r_a) || overlaps(r_out, r_b) || overlaps(r_out, r_o)) return GDG_EOVERLAP;

    DeviceInfo* dev = device_info(&st);
    if (!dev) return st;

    GemmParams& p = pl->p;
    std::memset(&p, 0, sizeof p);
    if (!encode_weight_3d(&p.tmA, args->b, E, N, K)) return GDG_ECUDA;
    for (int i = 0; i < 5; ++i)
        if (!encode_rows_2d(&p.tmB[i], args->a, rows, in_cols, 8u << i)) return GDG_ECUDA;
    p.offs = offs;
    p.out = args->out;
    p.partial = nullptr;
    p.err = dev->err;
    p.rows = rows;
    p.E = E;
    p.N = N;
    p.K = K;
    p.offs_kind = args->offs_kind;
    p.split_rows = 0;
    p.ld_out = L.ld;
    // Row tile (and ring geometry), from the shapes alone: groups of at most 64 rows on
    // average only stream weights, and a 128-row tile keeps more weight bytes in flight
    // (larger groups lose more to re-reading weight tiles than they gain).
    pl->rt = (rows <= static_cast<int64_t>(E) * 64) ? 128 : 256;
    const int64_t ft = (OP == gdg::OP_FWD) ? ceil_div(N, gdg::kPairM) : ceil_div(K, gdg::kPairM);
    const int64_t ub = ft * (ceil_div(rows, pl->rt) + E);
    if (ub > INT32_MAX) return GDG_EINVAL;
    p.max_units = static_cast<int>(ub);
    pl->grid = pair_grid(ub, dev->pairs);
    pl->launch = true;
    return GDG_OK;
}

// wgrad plan.  ordered = 0 selects the non-deterministic form: row chunks of the split form
// add their fp32 tiles into the destination with unordered atomic adds (no partials, no
// ordered reduce); the unsplit form runs in its fixed order either way.
gdg_status plan_wgrad(const gdg_args* args, const int32_t* offs, int E, int N, int K,
                      gdg_dtype out_dtype, int accumulate, Plan* pl, int ordered = 1) {
    gdg_status st = check_common(args, offs, E, N, K, out_dtype);
    if (st != GDG_OK) return st;
    if (accumulate != 0 && accumulate != 1) return GDG_EINVAL;
    int32_t split_rows = args->split_rows;
    if (split_rows < -1 || (split_rows > 0 && split_rows % 64 != 0)) return GDG_EINVAL;
    const int64_t rows = args->rows;
    if (!args->out) return GDG_EINVAL;
    if (rows > 0 && (!args->a || !args->b)) return GDG_EINVAL;
    if (!aligned16(args->out) || !aligned16(offs) || (rows > 0 && (!aligned16(args->a) ||
                                                                   !aligned16(args->b))))
        return GDG_EALIGN;
    const size_t osz = out_dtype == GDG_FP32 ? 4 : 2;
    OutLayout L;
    st = out_layout(args, N, K, E, osz, true, &L);
    if (st != GDG_OK) return st;
    const Range r_out = range_of(args->out, L.span);
    const Range r_a = range_of(args->a, static_cast<uint64_t>(rows) * N * 2);
    const Range r_b = range_of(args->b, static_cast<uint64_t>(rows) * K * 2);
    const Range r_o = range_of(offs, static_cast<uint64_t>(E + args->offs_kind) * 4);
    if (overlaps(r_out, r_o) || (rows > 0 && (overlaps(r_out, r_a) || overlaps(r_out, r_b))))
        return GDG_EOVERLAP;
    pl->op = GDG_OP_WGRAD;
    pl->launch = false;
    if (rows == 0 && accumulate) return GDG_OK;   // nothing to add; out is left unchanged

    if (split_rows == 0) split_rows = auto_split_rows(rows, E, N, K);
    if (rows == 0) split_rows = -1;   // overwrite with no rows: the plain form writes +0.0
    const bool split = split_rows > 0;
    int64_t max_units = static_cast<int64_t>(E) * tiles_per_expert(N, K);
    if (split) {
        max_units = split_max_units(rows, E, N, K, split_rows);
        // ordered: the fp32 partial tiles; unordered: the fp32 sums of a bf16 out (none for fp32)
        const size_t need = ordered ? static_cast<size_t>(max_units) * gdg::kPartialElems * sizeof(float)
                                    : (out_dtype == GDG_FP32 ? 0 : static_cast<size_t>(E) * N * K * 4);
        if (need > 0 && (!args->workspace || args->workspace_bytes < need)) return GDG_EWORKSPACE;
        if (need > 0 && !aligned16(args->workspace)) return GDG_EALIGN;
        const Range r_w = range_of(need > 0 ? args->workspace : nullptr, need);
        if (overlaps(r_w, r_out) || overlaps(r_w, r_o) ||
            (rows > 0 && (overlaps(r_w, r_a) || overlaps(r_w, r_b))))
            return GDG_EOVERLAP;
    }
    if (max_units * gdg::kPairM >= INT32_MAX) return GDG_EINVAL;   // TMA row coordinates

    DeviceInfo* dev = device_info(&st);
    if (!dev) return st;

    const int epi = accumulate ? (out_dtype == GDG_FP32 ? gdg::EPI_FP32_ACC : gdg::EPI_BF16_ACC)
                               : (out_dtype == GDG_FP32 ? gdg::EPI_FP32 : gdg::EPI_BF16);
    GemmParams& p = pl->p;
    std::memset(&p, 0, sizeof p);
    // With rows == 0 no copy is ever issued; the maps still need a valid shape.
    const int64_t map_rows = rows > 0 ? rows : 1;
    const void* a = rows > 0 ? args->a : args->out;
    const void* b = rows > 0 ? args->b : args->out;
    if (!encode_rows_2d(&p.tmA, a, map_rows, N, 128u) ||
        !encode_rows_2d(&p.tmB[0], b, map_rows, K, 128u) ||
        !encode_rows_2d(&p.tmTail[0], a, map_rows, N, 16u) ||
        !encode_rows_2d(&p.tmTail[1], b, map_rows, K, 16u))
        return GDG_ECUDA;
    p.offs = offs;
    p.out = args->out;
    p.partial = split ? static_cast<float*>(args->workspace) : nullptr;
    p.err = dev->err;
    p.rows = rows;
    p.E = E;
    p.N = N;
    p.K = K;
    p.offs_kind = args->offs_kind;
    p.split_rows = split ? split_rows : 0;
    p.max_units = static_cast<int>(max_units);
    p.ld_out = L.ld;
    p.es_out = L.es;
    p.sort_groups = split ? 0 : sort_groups_rule(rows, E);
    pl->grid = pair_grid(max_units, dev->pairs);
    p.teams = teams_rule(p.sort_groups, tiles_per_expert(N, K), pl->grid / 2);
    pl->epi = split ? static_cast<int>(gdg::EPI_PARTIAL) : epi;
    pl->launch = true;
    pl->reduce = split && ordered;
    const int64_t vec4 = static_cast<int64_t>(E) * N * K / 4;
    int64_t dgrid = ceil_div(vec4, gdg::kReduceThreads);
    if (dgrid > static_cast<int64_t>(dev->sms) * 8) dgrid = static_cast<int64_t>(dev->sms) * 8;
    if (split && !ordered) {
        // The unordered adds go into out itself (fp32) or into the fp32 workspace (bf16), which
        // starts at +0.0 unless an fp32 out is accumulated into.
        const bool f32 = out_dtype == GDG_FP32;
        pl->epi = gdg::EPI_RED;
        p.partial = nullptr;
        if (!f32) {
            p.out = args->workspace;
            p.ld_out = K;
            p.es_out = static_cast<int64_t>(N) * K;
        }
        pl->zero = !f32 || !accumulate;
        pl->z.out = p.out;
        pl->z.E = E;
        pl->z.N = N;
        pl->z.K = K;
        pl->z.ld_out = p.ld_out;
        pl->z.es_out = p.es_out;
        pl->finish = !f32;
        pl->f.out = args->out;
        pl->f.acc = static_cast<const float*>(args->workspace);
        pl->f.E = E;
        pl->f.N = N;
        pl->f.K = K;
        pl->f.epi = accumulate ? gdg::EPI_BF16_ACC : gdg::EPI_BF16;
        pl->f.ld_out = L.ld;
        pl->f.es_out = L.es;
        pl->rgrid = static_cast<int>(dgrid);
    }
    if (split && ordered) {
        ReduceParams& r = pl->r;
        r.offs = offs;
        r.partial = static_cast<const float*>(args->workspace);
        r.out = args->out;
        r.rows = rows;
        r.E = E;
        r.N = N;
        r.K = K;
        r.offs_kind = args->offs_kind;
        r.epi = epi;
        r.split_rows = split_rows;
        r.max_units = static_cast<int>(max_units);
        r.ld_out = L.ld;
        r.es_out = L.es;
        pl->rgrid = static_cast<int>(dgrid);
    }
    return GDG_OK;
}

gdg_status launch_plan(const Plan& pl, cudaStream_t s) {
    if (!pl.launch) return GDG_OK;
    // The launch status is read from this host thread's last-error slot: clear what an earlier,
    // unrelated call on the thread may have left there (a sticky error survives and is seen).
    cudaGetLastError();
    const GemmParams& p = pl.p;
    const int g = pl.grid;
    if (pl.zero) {
        gdg::zero_f32_kernel<<<pl.rgrid, gdg::kReduceThreads, 0, s>>>(pl.z);
        const gdg_status st = launch_status(cudaGetLastError());
        if (st != GDG_OK) return st;
    }
    if (pl.op == GDG_OP_FWD) {
        if (pl.rt == 128)
            gdg::grouped_gemm_kernel<gdg::OP_FWD, gdg::EPI_BF16, 128><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
        else
            gdg::grouped_gemm_kernel<gdg::OP_FWD, gdg::EPI_BF16, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
        return launch_status(cudaGetLastError());
    }
    if (pl.op == GDG_OP_DGRAD) {
        if (pl.rt == 128)
            gdg::grouped_gemm_kernel<gdg::OP_DGRAD, gdg::EPI_BF16, 128><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
        else
            gdg::grouped_gemm_kernel<gdg::OP_DGRAD, gdg::EPI_BF16, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
        return launch_status(cudaGetLastError());
    }
    switch (pl.epi) {
        case gdg::EPI_BF16:
            gdg::grouped_gemm_kernel<gdg::OP_WGRAD, gdg::EPI_BF16, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
            break;
        case gdg::EPI_FP32:
            gdg::grouped_gemm_kernel<gdg::OP_WGRAD, gdg::EPI_FP32, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
            break;
        case gdg::EPI_BF16_ACC:
            gdg::grouped_gemm_kernel<gdg::OP_WGRAD, gdg::EPI_BF16_ACC, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
            break;
        case gdg::EPI_FP32_ACC:
            gdg::grouped_gemm_kernel<gdg::OP_WGRAD, gdg::EPI_FP32_ACC, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
            break;
        case gdg::EPI_RED:
            gdg::grouped_gemm_kernel<gdg::OP_WGRAD, gdg::EPI_RED, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
            break;
        default:
            gdg::grouped_gemm_kernel<gdg::OP_WGRAD, gdg::EPI_PARTIAL, 256><<<g, gdg::kThreads, gdg::kGemmSmemBytes, s>>>(p);
            break;
    }
    gdg_status st = launch_status(cudaGetLastError());
    if (st != GDG_OK) return st;
    if (pl.finish) {
        gdg::finish_bf16_kernel<<<pl.rgrid, gdg::kReduceThreads, 0, s>>>(pl.f);
        return launch_status(cudaGetLastError());
    }
    if (!pl.reduce) return st;
    gdg::wgrad_reduce_kernel<<<pl.rgrid, gdg::kReduceThreads, 0, s>>>(pl.r);
    return launch_status(cudaGetLastError());
}

gdg_status make_plan(int op, const gdg_args* args, const int32_t* offs, int E, int N, int K,
                     gdg_dtype out_dtype, int accumulate, Plan* pl) {
    switch (op) {
        case GDG_OP_FWD: return plan_fwd_like<gdg::OP_FWD>(args, offs, E, N, K, out_dtype, accumulate, pl);
        case GDG_OP_DGRAD: return plan_fwd_like<gdg::OP_DGRAD>(args, offs, E, N, K, out_dtype, accumulate, pl);
        case GDG_OP_WGRAD: return plan_wgrad(args, offs, E, N, K, out_dtype, accumulate, pl);
    }
    return GDG_EINVAL;
}

gdg_status run(int op, const gdg_args* args, const int32_t* offs, int E, int N, int K,
               gdg_dtype out_dtype, int accumulate, void* stream) {
    Plan pl;
    const gdg_status st = make_plan(op, args, offs, E, N, K, out_dtype, accumulate, &pl);
    if (st != GDG_OK) return st;
    return launch_plan(pl, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

gdg_status grouped_det_gemm_fwd(const gdg_args* args, const int32_t* offs, int E, int N, int K,
                                gdg_dtype out_dtype, int accumulate, void* stream) {
    return run(GDG_OP_FWD, args, offs, E, N, K, out_dtype, accumulate, stream);
}

gdg_status grouped_det_gemm_dgrad(const gdg_args* args, const int32_t* offs, int E, int N,
                                  int K, gdg_dtype out_dtype, int accumulate, void* stream) {
    return run(GDG_OP_DGRAD, args, offs, E, N, K, out_dtype, accumulate, stream);
}

int32_t grouped_det_gemm_auto_split_rows(int64_t rows, int E, int N, int K) {
    if (E < 1 || N <= 0 || K <= 0 || N % 8 || K % 8 || rows < 0) return -1;
    return auto_split_rows(rows, E, N, K);
}

size_t grouped_det_gemm_workspace_bytes(int op, int64_t rows, int E, int N, int K,
                                        gdg_dtype out_dtype, int accumulate, int32_t split_rows) {
    if (E < 1 || E > GDG_MAX_EXPERTS || N <= 0 || K <= 0 || rows < 0 || N % 8 || K % 8 ||
        (out_dtype != GDG_BF16 && out_dtype != GDG_FP32) || op < GDG_OP_FWD || op > GDG_OP_WGRAD)
        return static_cast<size_t>(-1);
    (void)accumulate;
    if (op != GDG_OP_WGRAD) return 0;
    if (split_rows == 0) split_rows = auto_split_rows(rows, E, N, K);
    if (split_rows < 0 || rows == 0) return 0;
    if (split_rows % 64 != 0) return static_cast<size_t>(-1);
    return static_cast<size_t>(split_max_units(rows, E, N, K, split_rows)) * gdg::kPartialElems *
           sizeof(float);
}

gdg_status grouped_det_gemm_wgrad(const gdg_args* args, const int32_t* offs, int E, int N,
                                  int K, gdg_dtype out_dtype, int accumulate, void* stream) {
    return run(GDG_OP_WGRAD, args, offs, E, N, K, out_dtype, accumulate, stream);
}

gdg_status grouped_gemm_wgrad(const gdg_args* args, const int32_t* offs, int E, int N, int K,
                              gdg_dtype out_dtype, int accumulate, int deterministic, void* stream) {
    if (deterministic != 0) return GDG_EINVAL;
    Plan pl;
    const gdg_status st = plan_wgrad(args, offs, E, N, K, out_dtype, accumulate, &pl, 0);
    if (st != GDG_OK) return st;
    return launch_plan(pl, static_cast<cudaStream_t>(stream));
}

size_t grouped_gemm_wgrad_workspace_bytes(int64_t rows, int E, int N, int K, gdg_dtype out_dtype,
                                          int accumulate, int32_t split_rows) {
    if (E < 1 || E > GDG_MAX_EXPERTS || N <= 0 || K <= 0 || rows < 0 || N % 8 || K % 8 ||
        (out_dtype != GDG_BF16 && out_dtype != GDG_FP32))
        return static_cast<size_t>(-1);
    (void)accumulate;
    if (split_rows == 0) split_rows = auto_split_rows(rows, E, N, K);
    if (split_rows < 0 || rows == 0 || out_dtype == GDG_FP32) return 0;
    if (split_rows % 64 != 0) return static_cast<size_t>(-1);
    return static_cast<size_t>(E) * N * K * 4;
}

struct gdg_plan {
    Plan pl;
};

gdg_status gdg_plan_create(int op, const gdg_args* args, const int32_t* offs, int E, int N, int K,
                           gdg_dtype out_dtype, int accumulate, gdg_plan** plan) {
    if (!plan) return GDG_EINVAL;
    *plan = nullptr;
    gdg_plan* h = new (std::nothrow) gdg_plan;
    if (!h) return GDG_EINVAL;
    const gdg_status st = make_plan(op, args, offs, E, N, K, out_dtype, accumulate, &h->pl);
    if (st != GDG_OK) {
        delete h;
        return st;
    }
    *plan = h;
    return GDG_OK;
}

gdg_status gdg_test_withhold_first_stage(int op, const gdg_args* args, const int32_t* offs,
                                         int E, int N, int K, gdg_dtype out_dtype,
                                         int accumulate, void* stream) {
    Plan pl;
    const gdg_status st = make_plan(op, args, offs, E, N, K, out_dtype, accumulate, &pl);
    if (st != GDG_OK) return st;
    pl.p.test_withhold = 1;
    return launch_plan(pl, static_cast<cudaStream_t>(stream));
}

void gdg_test_set_max_pairs(int pairs) { g_max_pairs.store(pairs > 0 ? pairs : 0); }

gdg_status gdg_plan_launch(const gdg_plan* plan, void* stream) {
    if (!plan) return GDG_EINVAL;
    return launch_plan(plan->pl, static_cast<cudaStream_t>(stream));
}

void gdg_plan_destroy(gdg_plan* plan) { delete plan; }

const char* gdg_status_string(gdg_status status) {
    switch (status) {
        case GDG_OK: return "ok";
        case GDG_EINVAL: return "invalid argument";
        case GDG_EALIGN: return "shape or alignment rule violated (N % 8, K % 8, 16-byte pointers)";
        case GDG_EOVERLAP: return "output overlaps itself, an input, the offsets or the workspace";
        case GDG_EWORKSPACE: return "workspace missing or too small";
        case GDG_ECUDA: return "CUDA call failed";
        case GDG_ETIMEOUT: return "an in-kernel wait ran out";
    }
    return "unknown status";
}

gdg_status gdg_device_error_async(unsigned int* dst, void* stream) {
    if (!dst) return GDG_EINVAL;
    gdg_status st = GDG_OK;
    DeviceInfo* dev = device_info(&st);
    if (!dev) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dst, dev->err, sizeof(unsigned int), cudaMemcpyDefault, s) != cudaSuccess ||
        cudaMemsetAsync(dev->err, 0, sizeof(unsigned int), s) != cudaSuccess) {
        cudaGetLastError();
        return GDG_ECUDA;
    }
    return GDG_OK;
}

gdg_status gdg_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GDG_ECUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return GDG_ECUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess)
        return GDG_ECUDA;
    return v == 0 ? GDG_OK : GDG_ETIMEOUT;
}

}  // extern "C"

// ------------------------------------------------------------------ fixed-scratch wgrad
//
// Scratch for the split partials of grouped_det_gemm_wgrad_noalloc, for callers that cannot
// allocate device memory.  In host code the name below is only a host-side stand-in: its
// device address comes from cudaGetSymbolAddress, once per device, with that device current.

static __device__ __align__(256) float g_noalloc_scratch[GDG_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

struct NoAllocSlot {
    std::atomic<void*> ptr{nullptr};
    std::mutex mu;
};

NoAllocSlot g_noalloc[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (looked up on first use).
void* noalloc_scratch(gdg_status* st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *st = GDG_ECUDA;
        return nullptr;
    }
    NoAllocSlot& slot = g_noalloc[dev];
    void* p = slot.ptr.load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lock(slot.mu);
    p = slot.ptr.load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            *st = GDG_ECUDA;
            return nullptr;
        }
        slot.ptr.store(p, std::memory_order_release);
    }
    return p;
}

// split_rows for the fixed scratch when the caller passes 0: the automatic value if its partials
// fit, else the smallest multiple of 64 whose partials fit (the most parallel split that does),
// or -1 when even one chunk per group does not fit.  Partials: tpe * (ceil(rows / s) + E) tiles.
int32_t noalloc_split_rows(int64_t rows, int E, int N, int K) {
    const int64_t tpe = tiles_per_expert(N, K);
    const int64_t tiles = GDG_NOALLOC_SCRATCH_BYTES / (gdg::kPartialElems * sizeof(float));
    const int64_t chunks = tiles / tpe - E;          // most row chunks whose partials fit
    if (chunks < 1) return -1;
    const int32_t a = auto_split_rows(rows, E, N, K);
    if (a > 0 && ceil_div(rows, a) <= chunks) return a;
    int64_t s = ceil_div(ceil_div(rows > 0 ? rows : 1, chunks), 64) * 64;
    if (s > (int64_t{1} << 30)) return -1;
    return static_cast<int32_t>(s);
}

}  // namespace

extern "C" gdg_status grouped_det_gemm_wgrad_noalloc(const gdg_args* args, const int32_t* offs,
                                                     int E, int N, int K, gdg_dtype out_dtype,
                                                     int accumulate, void* stream) {
    if (!args || args->split_rows < 0) return GDG_EINVAL;
    if (E < 1 || E > GDG_MAX_EXPERTS || N <= 0 || K <= 0 || N % 8 || K % 8 || args->rows < 0 ||
        args->rows > GDG_MAX_ROWS)
        return GDG_EINVAL;
    int32_t split_rows = args->split_rows;
    if (split_rows == 0) {
        split_rows = noalloc_split_rows(args->rows, E, N, K);
        if (split_rows < 0) return GDG_EWORKSPACE;
    }
    const size_t need = grouped_det_gemm_workspace_bytes(GDG_OP_WGRAD, args->rows, E, N, K,
                                                         out_dtype, accumulate, split_rows);
    if (need == static_cast<size_t>(-1)) return GDG_EINVAL;
    if (need > GDG_NOALLOC_SCRATCH_BYTES) return GDG_EWORKSPACE;
    gdg_args a = *args;
    a.split_rows = split_rows;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (need > 0) {
        gdg_status st = GDG_OK;
        a.workspace = noalloc_scratch(&st);
        if (!a.workspace) return st;
        a.workspace_bytes = GDG_NOALLOC_SCRATCH_BYTES;
    }
    return grouped_det_gemm_wgrad(&a, offs, E, N, K, out_dtype, accumulate, stream);
}
