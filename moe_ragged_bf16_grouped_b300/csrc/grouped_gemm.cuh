// Ragged BF16 grouped GEMM kernels for sm_103a: fwd, dgrad and wgrad (plain, fused
// accumulate, or fixed split partials), plus the ordered reduce of those partials.
//
// Operations (computation table of the "Cake ragged BF16 grouped GEMM (experimental)"
// docs page; group e = rows [s_e, t_e) of the packed operands, intro paragraph):
//   fwd    Y[s_e:t_e]  = X[s_e:t_e] @ W[e]^T
//   dgrad  dX[s_e:t_e] = G[s_e:t_e] @ W[e]
//   wgrad  dW[e]       = G[s_e:t_e]^T @ X[s_e:t_e]
//
// Every GEMM kernel is persistent and runs as CTA pairs (clusters of two CTAs on two SMs):
// pair i walks work units u = i, i + pairs, ...  The unit list comes from the offsets on the
// device (no host sync): units are numbered group by group, each CTA counts them once, and
// every role keeps a cursor that walks the groups forward (reading offs) as u grows.
//
// MMA (tcgen05.mma.cta_group::2, M = 256 across the pair, N <= 256, K = 16 per instruction;
// each CTA holds 128 rows of A, half of the N rows of B, and its 128 rows of D in TMEM):
//   fwd    D[n, row] = sum_k  W[e][n][k] * X[row][k]   A = W  K-major,  B = X  K-major
//   dgrad  D[k, row] = sum_n  W[e][n][k] * G[row][n]   A = W  MN-major, B = G  K-major
//   wgrad  D[n, k]   = sum_r  G[r][n]    * X[r][k]     A = G  MN-major, B = X  MN-major
// For fwd / dgrad the packed rows are the MMA's N dimension, so a ragged group is
// covered with 16-row granularity (N = round_up(rows in tile, 16)) instead of the
// 128-row granularity of the M dimension; weights stream as the A operand.
// For wgrad the reduction runs over the group's rows in 128-row stages starting exactly
// at the group's first row.  A unit's last stage usually ends inside a 16-row MMA step: the
// ring stage serves only the whole steps, and the partial step is copied on its own (16 rows
// of each operand) into a small double-buffered tail buffer ahead of the unit's stages, where a
// "fixer" warp in each CTA zeroes the rows past the unit's end before the MMA reads it.
//
// Warp roles (384 threads per CTA): warp 0 lane 0 issues TMA loads of this CTA's halves
// into a kStages-deep ring, completing on the even CTA's "full" barriers, and the wgrad tail
// steps; warp 1 lane 0 of the even CTA issues the pair's MMAs into one of two TMEM accumulators
// (2 x 256 fp32 columns) and commits to the "empty" / "tmem full" barriers of both CTAs; warp 2
// owns the TMEM allocation; warp 3 of each CTA zeroes wgrad tail rows; warps 4..11 of both
// CTAs drain their TMEM rows (tcgen05.ld; two warps per 32-lane quarter, one per half of the
// columns) and write the outputs while the next tile's MMAs run into the other accumulator.
//
// Determinism: each output element is produced by exactly one CTA pair, whose MMA sequence
// is fixed by the unit's coordinates alone (never by the grid size or timing); the
// split form writes each partial once and the reduce adds partials in chunk order.
// No atomics touch the data.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace gdg {

constexpr int kPairM = 256;                 // MMA M across the CTA pair
constexpr int kBM = 128;                    // A rows (and D rows) per CTA
constexpr int kBN = 256;                    // MMA N (max)
constexpr int kBK = 128;                    // reduction elements per stage: two 64-wide blocks
constexpr int kABytes = kBM * kBK * 2;      // 32 KB: this CTA's 128 rows of A
constexpr int kRingBytes = 3 * (kABytes + (kBN / 2) * kBK * 2);   // 192 KB operand ring
constexpr int kMaxStages = 4;

// Ring geometry, by the fwd / dgrad row tile RT (packed rows per tile): RT = 256 gives 3
// stages of 64 KB (A 32 KB + B 32 KB per CTA); RT = 128 gives 4 stages of 48 KB (A 32 KB +
// B 16 KB), i.e. a third more weight bytes in flight per SM for weight-streaming shapes.
// wgrad always uses RT = 256 (its B half is 128 columns of X).
template <int RT>
struct Ring {
    static constexpr int kStages = RT == 256 ? 3 : 4;
    static constexpr int kBBytes = (RT / 2) * kBK * 2;      // this CTA's half of B
    static constexpr int kStageBytes = kABytes + kBBytes;
    static_assert(kStages * kStageBytes == kRingBytes, "ring geometries share 192 KB");
    static_assert(kStages <= kMaxStages, "barrier arrays");
};
constexpr int kSubBytes = 128 * 128;        // one 128-row block of 64 bf16 (128 B) per row
constexpr int kEpiWarps = 8;
constexpr int kEpiBoxBytes = 32 * 64;       // wgrad staging box per warp: 32 rows x 64 B
constexpr int kEpiBytes = kEpiWarps * kEpiBoxBytes;
constexpr int kTailSub = 16 * 128;          // wgrad tail step: one 64-column block, 16 rows
constexpr int kTailBytes = 4 * kTailSub;    // G blocks 0, 1 then X blocks 0, 1 of this CTA
constexpr int kTailBufs = 2;
constexpr int kThreads = 384;               // GEMM kernel: 4 role warps + 8 epilogue warps
constexpr int kReduceThreads = 256;
constexpr int kMaxE = 1024;
constexpr int kMaxSorted = 128;             // wgrad: groups walked by size need E <= this
constexpr int kMaxTeams = 32;               // wgrad teams (one warp computes the assignment)
constexpr int kTmemCols = 512;
constexpr int kPartialElems = kPairM * kBN; // fp32 elements per split partial tile
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // any single wait > 2 s is a hang
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr uint32_t kSuspendNs = 20000;             // sleep hint of a waiting thread
constexpr uint64_t kCopyDrainNs = 2000000ull;   // after an abort: copies in flight land by then

enum Op : int { OP_FWD = 0, OP_DGRAD = 1, OP_WGRAD = 2 };
// EPI_RED (non-deterministic split form): each row chunk's fp32 tile is added into an fp32
// destination with unordered atomic adds instead of being stored as a partial.
enum Epi : int { EPI_BF16 = 0, EPI_FP32 = 1, EPI_BF16_ACC = 2, EPI_FP32_ACC = 3, EPI_PARTIAL = 4,
                 EPI_RED = 5 };

constexpr unsigned kDevErrTimeout = 6u;

struct GemmParams {
    // Operand maps (bf16, 128-byte swizzle, zero fill past every extent).  Every copy brings
    // one 64-column block; a stage's two blocks land as consecutive sub-tiles.
    CUtensorMap tmA;        // fwd / dgrad: W {K, N, E} box {64, 128, 1};
                            // wgrad: G {N, rows} box {64, 128}
    CUtensorMap tmB[5];     // fwd: X {K, rows}, dgrad: G {N, rows}, box {64, 8 << i};
                            // wgrad: tmB[0] = X {K, rows} box {64, 128}
    CUtensorMap tmTail[2];  // wgrad tail steps: G {N, rows}, X {K, rows}, box {64, 16}
    const int32_t* offs;
    void* out;
    float* partial;         // wgrad split form: [max_units][256][256] fp32
    unsigned int* err;      // device error word
    int64_t rows;
    int E, N, K;
    int offs_kind;
    int split_rows;         // wgrad: > 0 selects the split form
    int max_units;          // units at or past this index are skipped
    int test_withhold;      // test only: pair 0's even CTA arms its first stage but copies nothing
    int64_t ld_out;         // out row stride (elements)
    int64_t es_out;         // wgrad: out expert stride (elements)
    int sort_groups;        // wgrad, unsplit, E <= kMaxSorted: walk the groups by size
    int teams;              // sort_groups and tiles per expert < pairs: team schedule (below)
};


struct SmemCtl {
    uint64_t full[kMaxStages];  // even CTA: both CTAs' copies of a stage have landed
    uint64_t empty[kMaxStages]; // both CTAs: the pair's MMAs have read the stage
    uint64_t tb_full[kTailBufs];    // both CTAs (wgrad): this CTA's tail step has landed
    uint64_t tb_fixed[kTailBufs];   // even CTA: both CTAs zeroed the tail step's extra rows
    uint64_t tb_empty[kTailBufs];   // both CTAs: the pair's MMA has read the tail step
    uint64_t tfull[2];          // both CTAs: the accumulator is complete
    uint64_t tempty[2];         // even CTA: all 16 epilogue warps of the pair drained it
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int64_t warp_tot[kThreads / 32];
    uint16_t order[kMaxSorted];  // sort_groups: the groups by decreasing size (ties: index)
    int32_t msize[kMaxSorted];   // sort_groups: the row count of order[i]
    uint8_t team_of[kMaxSorted]; // teams: the team that runs order[i]
};

constexpr size_t kGemmSmemBytes =
    1024 + static_cast<size_t>(kRingBytes) + kEpiBytes + kTailBufs * kTailBytes + sizeof(SmemCtl);

// ------------------------------------------------------------------ schedule

// Division of 0 <= n < 2^31 by a divisor d >= 1 fixed for the launch, by multiplication
// (Granlund and Montgomery, "Division by invariant integers using multiplication", 1994):
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(n, m) + n) >> l
// (the sum stays below 2^32 because umulhi(n, m) < n < 2^31).
struct FastDiv {
    uint32_t d, m, l;
    __host__ __device__ static FastDiv make(uint32_t d) {
        FastDiv f;
        f.d = d;
        f.l = 0;
        while ((1ull << f.l) < d) ++f.l;
        f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
        return f;
    }
    __host__ __device__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
        return (__umulhi(n, m) + n) >> l;
#else
        return static_cast<uint32_t>(((static_cast<uint64_t>(n) * m >> 32) + n) >> l);
#endif
    }
};

struct Shape {
    int ft;     // feature tiles (fwd, dgrad) or tiles per expert (wgrad), 256 wide
    int kt;     // wgrad: k tiles per expert
    FastDiv ft_div, kt_div;   // wgrad: division by ft and by kt in the unit decode
};

template <int OP>
__device__ __forceinline__ Shape unit_shape(const GemmParams& p) {
    Shape s;
    if (OP == OP_FWD) { s.ft = (p.N + kPairM - 1) / kPairM; s.kt = 1; }
    else if (OP == OP_DGRAD) { s.ft = (p.K + kPairM - 1) / kPairM; s.kt = 1; }
    else { s.kt = (p.K + kBN - 1) / kBN; s.ft = ((p.N + kPairM - 1) / kPairM) * s.kt; }
    s.ft_div = FastDiv::make(static_cast<uint32_t>(s.ft));
    s.kt_div = FastDiv::make(static_cast<uint32_t>(s.kt));
    return s;
}

// The offsets that bound group e: its first row a and its end b, as stored.
__device__ __forceinline__ void group_raw(const int32_t* offs, int kind, int e, int32_t& a,
                                          int32_t& b) {
    if (kind == 0) { a = e > 0 ? __ldg(offs + e - 1) : 0; b = __ldg(offs + e); }
    else { a = __ldg(offs + e); b = __ldg(offs + e + 1); }
}

// Rows [s, s + m) of a group bounded by a and b, clamped to [0, rows]; a reversed range is
// empty.
__device__ __forceinline__ void group_clamp(int64_t a, int64_t b, int64_t rows, int& s, int& m) {
    a = a < 0 ? 0 : (a > rows ? rows : a);
    b = b < 0 ? 0 : (b > rows ? rows : b);
    if (b < a) b = a;
    s = static_cast<int>(a);
    m = static_cast<int>(b - a);
}

// Rows [s, s + m) of group e.
__device__ __forceinline__ void group_range(const int32_t* offs, int kind, int64_t rows, int e,
                                            int& s, int& m) {
    int32_t a, b;
    group_raw(offs, kind, e, a, b);
    group_clamp(a, b, rows, s, m);
}

// Units of a group of m rows.  64-bit: with offsets that are not cumulative (several groups
// clamped to the same rows) the sum over groups can pass the int range, and m + RT - 1 can pass
// it for m near 2^31.  A single group's count never exceeds max_units (< 2^31), checked on the
// host.
template <int OP, int RT>
__device__ __forceinline__ int64_t units_of_group(int m, const Shape& sh, int split_rows) {
    if (OP == OP_WGRAD) {
        if (split_rows > 0)
            return ((static_cast<int64_t>(m) + split_rows - 1) / split_rows) * sh.ft;
        return sh.ft;       // every tile of every expert, empty groups included
    }
    return ((static_cast<int64_t>(m) + RT - 1) / RT) * sh.ft;
}

// Builds start/size/prefix/total in shared memory (ordered reduce of split partials).  Every
// thread of the block (kReduceThreads) calls it.
template <int OP>
__device__ void build_schedule(const int32_t* offs, int kind, int64_t rows, int E,
                               int split_rows, int max_units, const Shape& sh, int* start,
                               int* size, int* prefix, int64_t* warp_tot, int* total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Each count is capped at max_units (< 2^31), so no 64-bit partial sum below can overflow;
    // prefixes are capped at max_units again when stored (no unit at or past max_units exists).
    int64_t v[4], local = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int e = tid * 4 + j;
        v[j] = 0;
        if (e < E) {
            int s, m;
            group_range(offs, kind, rows, e, s, m);
            start[e] = s;
            size[e] = m;
            const int64_t n = units_of_group<OP, 256>(m, sh, split_rows);
            v[j] = n < max_units ? n : max_units;
        }
        local += v[j];
    }
    int64_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t t = lane < kReduceThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kReduceThreads / 32) warp_tot[lane] = t;
    }
    __syncthreads();
    int64_t base = (warp ? warp_tot[warp - 1] : 0) + x - local;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int e = tid * 4 + j;
        if (e < E) prefix[e] = static_cast<int>(base < max_units ? base : max_units);
        base += v[j];
    }
    if (tid == 0) {
        const int64_t tot = warp_tot[kReduceThreads / 32 - 1];
        prefix[E] = static_cast<int>(tot < max_units ? tot : max_units);
        *total = prefix[E];
    }
    __syncthreads();
}

// Number of work units over all groups, capped at max_units.  Every thread of the block
// calls it.
template <int OP, int RT>
__device__ int count_units(const GemmParams& p, const Shape& sh, int64_t* warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t local = 0;      // at most 3 groups per thread, each below 2^31 units
    for (int e = tid; e < p.E; e += kThreads) {
        int s, m;
        group_range(p.offs, p.offs_kind, p.rows, e, s, m);
        local += units_of_group<OP, RT>(m, sh, p.split_rows);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if (lane == 0) warp_tot[warp] = local;
    __syncthreads();
    int64_t tot = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += warp_tot[w];
    return static_cast<int>(tot < p.max_units ? tot : p.max_units);
}

// Walks the groups forward: the pos-th group of the walk is e (e = pos, or order[pos] when the
// groups are walked by size); it holds units [base, base + n) and rows [s, s + m).  base and n
// are 64-bit for the same reason as units_of_group.
struct Cursor {
    int64_t base, n;
    int pos, e, s, m;
    int32_t na, nb, na2, nb2;   // the offsets of the walk's next two groups, loaded ahead
    const uint16_t* order;      // nullptr: natural order
};

// sort_groups: order[] = the groups by decreasing row count, ties by index.  Long groups first
// and groups of similar length next to each other keep the pairs that share a group's rows
// (every tile of it) working on them at the same time, so the rows are read from HBM once.
// Every thread of the block calls it; a later __syncthreads publishes order[].
__device__ __forceinline__ void sort_groups_by_size(const GemmParams& p, uint16_t* order,
                                                   int32_t* msize) {
    for (int e = threadIdx.x; e < p.E; e += kThreads) {
        int s, m;
        group_range(p.offs, p.offs_kind, p.rows, e, s, m);
        int rank = 0;
        for (int j = 0; j < p.E; ++j) {
            int sj, mj;
            group_range(p.offs, p.offs_kind, p.rows, j, sj, mj);
            rank += (mj > m || (mj == m && j < e)) ? 1 : 0;
        }
        order[rank] = static_cast<uint16_t>(e);
        msize[rank] = m;
    }
}

// Team schedule (wgrad, groups walked by size, T = tiles per expert below the pair count P):
// the pairs form floor(P / T) full teams of T pairs, which run each of their groups as one
// round (pair i of the team takes tile i), and, if P is not a multiple of T, a remainder team
// of b = P mod T pairs, which runs each of its groups in ceil(T / b) rounds.  Every tile of a
// group is then in flight at the same time (full team) or within one round (remainder team),
// so the group's rows of G and X are read from HBM about once, where dealing units to the
// pairs in turn spreads a group's tiles over pairs that reach them at different times.  Groups
// go, largest first, to the team that would finish them first (modelled time: rounds x
// (rows / 128 + 1.5) stages; ties to the lower team).  Every CTA computes the same
// assignment; warp 0 calls it, lane q holding team q.
__device__ void assign_teams(int E, int T, int P, const int32_t* msize, uint8_t* team_of) {
    const int lane = threadIdx.x & 31;
    const int full = P / T, b = P - full * T;
    const int nteams = full + (b > 0 ? 1 : 0);
    const float rounds = lane < full ? 1.f : static_cast<float>((T + b - 1) / max(b, 1));
    float fin = 0.f;
    for (int i = 0; i < E; ++i) {
        const float cost = rounds * (static_cast<float>(msize[i]) * (1.f / 128.f) + 1.5f);
        float v = lane < nteams ? fin + cost : 3.0e38f;
        int who = lane;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int w2 = __shfl_xor_sync(0xffffffffu, who, o);
            if (v2 < v || (v2 == v && w2 < who)) { v = v2; who = w2; }
        }
        if (lane == who) fin += cost;
        if (lane == 0) team_of[i] = static_cast<uint8_t>(who);
    }
}

// Issues the loads of the offsets of the walk's group pos + d (if any); their values are first
// used when the cursor reaches that group, so the load latency is hidden (two groups ahead: one
// unit step may cross two short groups).
__device__ __forceinline__ void cursor_load(Cursor& cu, const GemmParams& p, int d, int32_t& a,
                                            int32_t& b) {
    if (cu.pos + d < p.E) {
        const int e = cu.order ? cu.order[cu.pos + d] : cu.pos + d;
        group_raw(p.offs, p.offs_kind, e, a, b);
    }
}

template <int OP, int RT>
__device__ __forceinline__ void cursor_init(Cursor& cu, const GemmParams& p, const Shape& sh,
                                            const uint16_t* order) {
    cu.order = order;
    cu.pos = 0;
    cu.e = order ? order[0] : 0;
    cu.base = 0;
    group_range(p.offs, p.offs_kind, p.rows, cu.e, cu.s, cu.m);
    cu.n = units_of_group<OP, RT>(cu.m, sh, p.split_rows);
    cursor_load(cu, p, 1, cu.na, cu.nb);
    cursor_load(cu, p, 2, cu.na2, cu.nb2);
}

// Moves the cursor to the group that holds unit u (u never decreases between calls, and
// u < total, so the last group is never passed).
template <int OP, int RT>
__device__ __forceinline__ void cursor_seek(Cursor& cu, const GemmParams& p, const Shape& sh,
                                            int u) {
    while (u >= cu.base + cu.n && cu.pos + 1 < p.E) {
        cu.base += cu.n;
        ++cu.pos;
        cu.e = cu.order ? cu.order[cu.pos] : cu.pos;
        group_clamp(cu.na, cu.nb, p.rows, cu.s, cu.m);
        cu.n = units_of_group<OP, RT>(cu.m, sh, p.split_rows);
        cu.na = cu.na2;
        cu.nb = cu.nb2;
        cursor_load(cu, p, 2, cu.na2, cu.nb2);
    }
}

// fp32 weight gradients of long groups: the tensor core's fp32 accumulator drifts by about
// 0.7 ulp per MMA step, so a group longer than kChunkStages stages (2048 rows) is reduced in
// chunks of that many rows, each accumulated fresh in one TMEM buffer and added (fp32,
// round to nearest even, in chunk order) into a running sum kept in the other TMEM buffer.
constexpr int kChunkStages = 16;

// Per TMEM buffer, in registers: on the MMA issuer, the uses of the buffer so far, each ended
// by one tempty phase; on the epilogue warps, the tfull phases of the buffer waited for so far.
// The two differ by the running-sum uses of chunked units, which the epilogue warps take
// without a tfull phase.
struct Acq {
    uint32_t n0 = 0, n1 = 0;
    __device__ __forceinline__ uint32_t of(int b) const { return b ? n1 : n0; }
    __device__ __forceinline__ void bump(int b) {
        if (b) ++n1;
        else ++n0;
    }
};

template <int OP, int EPI>
__device__ __forceinline__ int chunks_of(int nkb) {
    constexpr bool chunked =
        OP == OP_WGRAD &&
        (EPI == EPI_FP32 || EPI == EPI_FP32_ACC || EPI == EPI_PARTIAL || EPI == EPI_RED);
    if (!chunked || nkb <= kChunkStages) return 1;
    return (nkb + kChunkStages - 1) / kChunkStages;
}

// wgrad: a unit whose rows end inside a 16-row MMA step (rows of another group or split
// follow in that step).  Its last ring stage serves only the whole 16-row steps; the partial
// step is loaded on its own into a tail buffer, one unit ahead, where both CTAs zero the rows
// past the unit's end before the MMA reads it.  Returns the rows of the last stage, or 0 when
// the unit has no partial step.
__device__ __forceinline__ int tail_rows(int nred, int nkb) {
    if (nkb <= 0) return 0;
    const int v = nred - (nkb - 1) * kBK;
    return (v & 15) != 0 ? v : 0;
}


struct Tile {
    int e;
    int f0;      // first M index of the pair tile (fwd: n, dgrad: k, wgrad: n)
    int c0;      // first N index (fwd/dgrad: packed row, wgrad: k)
    int ncols;   // valid N extent (<= 256)
    int r0;      // wgrad: first reduction row
    int nred;    // reduction length (fwd: K, dgrad: N, wgrad: rows of this unit)
    int nkb;     // 64-wide reduction stages
    int u;
};

template <int OP, int RT>
__device__ __forceinline__ Tile decode_unit(const GemmParams& p, Cursor& cu, const Shape& sh,
                                            int u) {
    cursor_seek<OP, RT>(cu, p, sh, u);
    Tile t;
    t.u = u;
    t.e = cu.e;
    const int local = static_cast<int>(u - cu.base);   // < cu.n, which fits an int
    const int s = cu.s, m = cu.m;
    if (OP == OP_WGRAD) {
        const int sp = static_cast<int>(sh.ft_div.div(static_cast<uint32_t>(local)));
        const int rem = local - sp * sh.ft;
        const int nt = static_cast<int>(sh.kt_div.div(static_cast<uint32_t>(rem)));
        const int kt = rem - nt * sh.kt;
        t.f0 = nt * kPairM;
        t.c0 = kt * kBN;
        t.ncols = min(kBN, p.K - t.c0);
        if (p.split_rows > 0) {
            t.r0 = s + sp * p.split_rows;
            t.nred = min(p.split_rows, m - sp * p.split_rows);
        } else {
            t.r0 = s;
            t.nred = m;
        }
    } else {
        const int rc_n = static_cast<int>((static_cast<int64_t>(m) + RT - 1) / RT);
        const int ft = local / rc_n, rc = local - ft * rc_n;
        t.f0 = ft * kPairM;
        t.c0 = s + rc * RT;
        t.ncols = min(RT, m - rc * RT);
        t.r0 = 0;
        t.nred = (OP == OP_FWD) ? p.K : p.N;
    }
    t.nkb = (t.nred + kBK - 1) / kBK;
    return t;
}

// The units of one CTA pair, in the order it runs them: units pair, pair + pairs, ... of the
// group-by-group numbering (decode_unit), or, with teams, the tiles of the groups its team
// runs.  Every role of both CTAs walks the same sequence.
struct Walker {
    Cursor cu;
    int u, pair, npairs, total;
    bool teams;
    const SmemCtl* c;
    int my_team, slot, tsize, rounds, last;   // team geometry (tsize = pairs of the team)
    int pos, e, s, m, r, off, npos, walk;
    int32_t na, nb;                           // offsets of the team's next group, loaded ahead
};

// The order in which a team visits the size-sorted list: step j of the walk looks at position
// walk_pos(j).  A full team alternates between the largest and the smallest groups left
// (kWalkAlternate), so that the epilogue writes out a short group's tiles while the MMAs of a
// long group run; the remainder team goes from the smallest group up (kWalkAscending), so that
// its output writes fall while the full teams run long groups.  The order changes only when a
// tile runs, never what it computes.
enum Walk : int { kWalkAlternate = 0, kWalkAscending = 1 };

__device__ __forceinline__ int walk_pos(int j, int E, int walk) {
    if (walk == kWalkAscending) return E - 1 - j;
    return (j & 1) ? E - 1 - (j >> 1) : (j >> 1);
}

// The first step at or after from whose group belongs to the team (E if none).
__device__ __forceinline__ int team_next(const SmemCtl* c, int E, int team, int from, int walk) {
    while (from < E && c->team_of[walk_pos(from, E, walk)] != team) ++from;
    return from;
}

template <int OP, int RT>
__device__ __forceinline__ void walker_init(Walker& w, const GemmParams& p, const Shape& sh,
                                            const SmemCtl* c, bool sorted, int pair, int npairs,
                                            int total) {
    w.u = pair;
    w.pair = pair;
    w.npairs = npairs;
    w.total = total;
    w.c = c;
    w.teams = OP == OP_WGRAD && sorted && p.teams;
    if (!w.teams) {
        cursor_init<OP, RT>(w.cu, p, sh, sorted ? c->order : nullptr);
        return;
    }
    const int T = sh.ft, full = npairs / T, b = npairs - full * T;
    w.my_team = pair / T;                      // == full for the remainder team
    w.slot = pair - w.my_team * T;
    w.tsize = w.my_team < full ? T : b;
    w.rounds = w.my_team < full ? 1 : (T + b - 1) / b;
    w.last = T - (w.rounds - 1) * w.tsize;     // tiles in the last round
    w.off = 0;
    w.r = w.rounds;                            // no group yet
    w.pos = -1;
    w.walk = w.my_team < full ? kWalkAlternate : kWalkAscending;
    w.npos = team_next(c, p.E, w.my_team, 0, w.walk);
    if (w.npos < p.E) group_raw(p.offs, p.offs_kind, c->order[walk_pos(w.npos, p.E, w.walk)], w.na, w.nb);
}

template <int OP, int RT>
__device__ __forceinline__ bool walker_next(Walker& w, const GemmParams& p, const Shape& sh,
                                            Tile& t) {
    if (!w.teams) {
        if (w.u >= w.total) return false;
        t = decode_unit<OP, RT>(p, w.cu, sh, w.u);
        w.u += w.npairs;
        return true;
    }
    for (;;) {
        if (w.r < w.rounds) {
            // Round r: the team's slots take tiles r * tsize + (slot - off) mod tsize; in the last
            // round only the first `last` of them exist.  off turns by `last` from one group to
            // the next, so the idle slots of the remainder team take turns.
            int s2 = w.slot - w.off;
            if (s2 < 0) s2 += w.tsize;
            const int tile = w.r * w.tsize + s2;
            ++w.r;
            if (tile >= sh.ft) continue;
            const int nt = static_cast<int>(sh.kt_div.div(static_cast<uint32_t>(tile)));
            const int kt = tile - nt * sh.kt;
            t.u = -1;
            t.e = w.e;
            t.f0 = nt * kPairM;
            t.c0 = kt * kBN;
            t.ncols = min(kBN, p.K - t.c0);
            t.r0 = w.s;
            t.nred = w.m;
            t.nkb = (t.nred + kBK - 1) / kBK;
            return true;
        }
        if (w.pos >= 0) {                      // the team's next group: turn the idle slots
            w.off += w.last;
            if (w.off >= w.tsize) w.off -= w.tsize;
        }
        w.pos = w.npos;
        if (w.pos >= p.E) return false;
        w.e = w.c->order[walk_pos(w.pos, p.E, w.walk)];
        group_clamp(w.na, w.nb, p.rows, w.s, w.m);
        w.npos = team_next(w.c, p.E, w.my_team, w.pos + 1, w.walk);
        if (w.npos < p.E)
            group_raw(p.offs, p.offs_kind, w.c->order[walk_pos(w.npos, p.E, w.walk)], w.na, w.nb);
        w.r = 0;
    }
}

// fwd / dgrad: MMA N (rows of the tile rounded up to 16), each CTA's half of it, and the
// index i of the smallest row box (8 << i rows) that holds that half.
__device__ __forceinline__ void row_split(int ncols, int& n_mma, int& half, int& bi) {
    n_mma = (ncols + 15) & ~15;
    half = n_mma >> 1;
    bi = 0;
    while ((8 << bi) < half) ++bi;
}

// ------------------------------------------------------------------ waits

struct Pair {
    uint32_t rank;        // 0 (even CTA: issues the MMAs) or 1
    uint32_t peer_abort;  // shared::cluster address of the other CTA's abort flag
};

__device__ __forceinline__ void raise_abort(SmemCtl* c, const Pair& pr, unsigned int* err) {
    *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
    st_cluster_u32(pr.peer_abort, 1u);
    atomicCAS(err, 0u, kDevErrTimeout);
}

// Bounded wait on an mbarrier phase (cluster-scope acquire).  Gives up when either CTA of
// the pair has aborted, or after kWaitLimitNs, in which case it raises the abort flag of
// both CTAs and records a timeout.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, SmemCtl* c,
                                         const Pair& pr, unsigned int* err) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity, kSuspendNs)) return true;
        if (*reinterpret_cast<volatile int*>(&c->abort_flag)) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            raise_abort(c, pr, err);
            return false;
        }
    }
}

// Lane 0 waits (bounded); __syncwarp then orders the rest of the warp after its acquire,
// so the other lanes need not poll the barrier themselves.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, SmemCtl* c,
                                              const Pair& pr, unsigned int* err) {
    const int lane = threadIdx.x & 31;
    int ok = 1;
    if (lane == 0) ok = wait_bar(bar, parity, c, pr, err);
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait that ignores the abort flag: used to let in-flight copies and MMAs land
// before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainLimitNs) break;
    }
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

// ------------------------------------------------------------------ epilogue helpers

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Descriptor address-field offsets (bytes / 16) of MMA step kk (K = 16) within a stage.
// K-major operands (fwd A, fwd / dgrad B): 16-element steps are 32 B apart inside a 64-wide
// block and blocks are a sub-tile apart (A: kSubBytes; B: b_sub).  MN-major operands (dgrad A,
// wgrad A and B): 16 reduction rows are 2 KB apart.
template <int OP>
__device__ __forceinline__ uint64_t a_step(int kk) {
    return OP == OP_FWD ? static_cast<uint64_t>((kk >> 2) * (kSubBytes >> 4) + (kk & 3) * 2)
                        : static_cast<uint64_t>(kk * (2048 >> 4));
}

template <int OP>
__device__ __forceinline__ uint64_t b_step(int kk, uint32_t b_sub) {
    return OP == OP_WGRAD ? static_cast<uint64_t>(kk * (2048 >> 4))
                          : static_cast<uint64_t>((kk >> 2) * (b_sub >> 4) + (kk & 3) * 2);
}

// ------------------------------------------------------------------ the GEMM kernel

// EPI: the epilogue (fwd / dgrad: EPI_BF16; wgrad: any, EPI_PARTIAL for the split form).
// RT: the fwd / dgrad row tile, which also picks the ring geometry (wgrad: 256).
template <int OP, int EPI, int RT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // Same offset in both CTAs of the pair: the MMA reads A and B of both at one address.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    using R = Ring<RT>;
    uint8_t* stage_area = smem + kRingBytes;                 // wgrad epilogue staging boxes
    uint8_t* tail_area = stage_area + kEpiBytes;              // wgrad tail-step buffers
    SmemCtl* c = reinterpret_cast<SmemCtl*>(tail_area + kTailBufs * kTailBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Shape sh = unit_shape<OP>(p);
    Pair pr;
    pr.rank = cluster_ctarank();
    pr.peer_abort = mapa_shared(smem_u32(&c->abort_flag), pr.rank ^ 1u);
    const bool even = pr.rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

    if (tid == 0) {
        for (int s = 0; s < R::kStages; ++s) {
            mbar_init(&c->full[s], 1);
            mbar_init(&c->empty[s], 1);
        }
        for (int b = 0; b < kTailBufs; ++b) {
            mbar_init(&c->tb_full[b], 1);
            mbar_init(&c->tb_fixed[b], 2);   // one arrival per CTA's fixer
            mbar_init(&c->tb_empty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c->tfull[b], 1);
            mbar_init(&c->tempty[b], 2 * kEpiWarps);   // one arrival per epilogue warp of the pair
        }
        mbar_init(&c->drain, 1);
        c->abort_flag = 0;
        fence_mbar_init();
    }
    if (tid == 32) {
        prefetch_tmap(&p.tmA);
        if (OP == OP_WGRAD) {
            prefetch_tmap(&p.tmB[0]);
        } else
            for (int i = 0; i < 5; ++i) prefetch_tmap(&p.tmB[i]);
    }
    const bool sorted = OP == OP_WGRAD && p.sort_groups && p.E <= kMaxSorted;
    if (sorted) sort_groups_by_size(p, c->order, c->msize);
    const int total = count_units<OP, RT>(p, sh, c->warp_tot);   // its __syncthreads publishes order
    if (sorted && p.teams && warp == 0) assign_teams(p.E, sh.ft, npairs, c->msize, c->team_of);
    // Both CTAs' barriers are initialised (and the peer has started) before any CTA signals
    // the other's barriers or allocates TMEM together with it; the cluster barrier also
    // publishes the team assignment to the CTA's threads.
    cluster_sync();
    Walker wk;
    walker_init<OP, RT>(wk, p, sh, c, sorted, pair, npairs, total);
    if (warp == 2) {
        tmem_alloc_pair(&c->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = c->tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full0 = mapa_shared(smem_u32(&c->full[0]), 0u);
            int stage = 0, jt = 0;   // jt: units with a tail step so far
            uint32_t phase = 0;
            bool ok = true;
            Tile t;
            for (int j = 0; ok && walker_next<OP, RT>(wk, p, sh, t); ++j) {
                int n_mma = 0, half = 0, bi = 0;
                if (OP != OP_WGRAD) row_split(t.ncols, n_mma, half, bi);
                const uint32_t bytes = (OP == OP_WGRAD)
                                           ? 2u * (kABytes + R::kBBytes)
                                           : 2u * (kABytes + (8u << bi) * 256u);
                const int fa = t.f0 + kBM * static_cast<int>(pr.rank);   // this CTA's A rows
                if (OP == OP_WGRAD) {
                    const int v = tail_rows(t.nred, t.nkb);
                    if (v) {
                        // The unit's partial 16-row step, into its tail buffer (own barrier),
                        // ahead of the unit's ring stages.
                        const int tb = jt & 1;
                        if (!wait_bar(&c->tb_empty[tb], ((jt >> 1) & 1) ^ 1u, c, pr, p.err)) {
                            ok = false;
                            break;
                        }
                        const int rt0 = t.r0 + (t.nkb - 1) * kBK + (v & ~15);
                        const int xb = (t.c0 + (kBN / 2) * static_cast<int>(pr.rank));
                        uint8_t* tbuf = tail_area + tb * kTailBytes;
                        mbar_arrive_expect_tx(&c->tb_full[tb], kTailBytes);
                        tma_load_2d(tbuf, &p.tmTail[0], &c->tb_full[tb], fa, rt0);
                        tma_load_2d(tbuf + kTailSub, &p.tmTail[0], &c->tb_full[tb], fa + 64, rt0);
                        tma_load_2d(tbuf + 2 * kTailSub, &p.tmTail[1], &c->tb_full[tb], xb, rt0);
                        tma_load_2d(tbuf + 3 * kTailSub, &p.tmTail[1], &c->tb_full[tb], xb + 64, rt0);
                        ++jt;
                    }
                }
                for (int kb = 0; kb < t.nkb; ++kb) {
                    if (!wait_bar(&c->empty[stage], phase ^ 1u, c, pr, p.err)) { ok = false; break; }
                    uint8_t* a = smem + stage * R::kStageBytes;
                    uint8_t* b = a + kABytes;
                    const uint32_t fb = full0 + stage * 8u;
                    if (even) mbar_arrive_expect_tx(&c->full[stage], bytes);
                    // Failure-detection test: the stage's barrier never completes, so the MMA
                    // issuer's bounded wait runs out and the pair aborts.
                    if (p.test_withhold && pair == 0 && even && j == 0 && kb == 0) {
                        if (++stage == R::kStages) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    // Two copies per operand and stage, one per 64-column block, landing as
                    // consecutive sub-tiles.  Columns and rows past a tensor's extent read as
                    // zeros, so N and K need not be multiples of the tile (every x coordinate
                    // is a multiple of 64 elements).
                    const int kx = kb * kBK;
                    if (OP == OP_FWD || OP == OP_DGRAD) {
                        // fwd A: 128 n-rows of W[e] from fa x k columns kx, kx + 64.
                        // dgrad A: n-rows kx.. of W[e] x this CTA's k columns fa, fa + 64.
                        const int ax = OP == OP_FWD ? kx : fa, ay = OP == OP_FWD ? fa : kx;
                        tma_load_3d_pair(a, &p.tmA, fb, ax, ay, t.e);
                        tma_load_3d_pair(a + kSubBytes, &p.tmA, fb, ax + 64, ay, t.e);
                        // B: packed rows of this CTA's half x the stage's reduction columns.
                        const int rb = t.c0 + half * static_cast<int>(pr.rank);
                        tma_load_2d_pair(b, &p.tmB[bi], fb, kx, rb);
                        tma_load_2d_pair(b + (8 << bi) * 128, &p.tmB[bi], fb, kx + 64, rb);
                    } else {
                        // 128 reduction rows x this CTA's two 64-wide blocks of G and of X.
                        const int r = t.r0 + kb * kBK;
                        const int xb = t.c0 + (kBN / 2) * static_cast<int>(pr.rank);
                        tma_load_2d_pair(a, &p.tmA, fb, fa, r);
                        tma_load_2d_pair(a + kSubBytes, &p.tmA, fb, fa + 64, r);
                        tma_load_2d_pair(b, &p.tmB[0], fb, xb, r);
                        tma_load_2d_pair(b + kSubBytes, &p.tmB[0], fb, xb + 64, r);
                    }
                    if (++stage == R::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            // After an abort, let every copy this thread started land before the CTA exits.
            // Most complete on the even CTA's barriers, which this CTA cannot observe, so it
            // waits a fixed time that covers any copy in flight.
            if (!ok) spin_ns(kCopyDrainNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer (even CTA)
        // One thread waits, issues and commits; the other lanes of the warp stay idle.
        // TMEM buffers alternate between units; acq counts the uses of each buffer (its
        // tempty phases).  A chunked unit keeps buffer A for its chunks and leaves buffer B to
        // the epilogue warps for the running sum.
        if (even && lane == 0) {
            int stage = 0, nextb = 0, jt = 0;   // jt: units with a tail step so far
            uint32_t phase = 0;
            Acq acq;
            bool ok = true;
            Tile t;
            while (ok && walker_next<OP, RT>(wk, p, sh, t)) {
                const int nch = chunks_of<OP, EPI>(t.nkb);
                const int A = nextb, B = nextb ^ 1;
                if (nch > 1) {
                    // The running sum is a use of B that no MMA writes: the epilogue warps
                    // start it once they are done with B's previous use (each warp touches only
                    // its own lanes and columns, in order), so the chunks' MMAs need not wait
                    // for that use to drain.  Its end is a tempty[B] phase like any other.  By
                    // the time this thread waits on tempty[B] again, the phase before this use
                    // has completed: chunk 1 waits for chunk 0's fold, which every epilogue
                    // warp starts only after it has released B's previous use.
                    acq.bump(B);
                }
                int n_mma = kBN, half = 0, bi = 0;
                if (OP != OP_WGRAD) row_split(t.ncols, n_mma, half, bi);
                const uint32_t idesc = idesc_bf16(kPairM, static_cast<uint32_t>(n_mma),
                                                  OP != OP_FWD, OP == OP_WGRAD);
                // MN-major operands: the two 64-wide M/N blocks are kSubBytes apart (LBO).
                const uint32_t b_sub = static_cast<uint32_t>((8 << bi) * 128);
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(A * kBN);
                const int tv = (OP == OP_WGRAD) ? tail_rows(t.nred, t.nkb) : 0;
                for (int ch = 0; ch < nch && ok; ++ch) {
                    if (!wait_bar(&c->tempty[A], (acq.of(A) & 1u) ^ 1u, c, pr, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const int kb0 = ch * kChunkStages;
                    const int kb1 = nch > 1 ? min(t.nkb, kb0 + kChunkStages) : t.nkb;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!wait_bar(&c->full[stage], phase, c, pr, p.err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * R::kStageBytes);
                        const uint32_t b_addr = a_addr + kABytes;
                        const int valid = t.nred - kb * kBK;
                        // fwd / dgrad: a last stage of 64 (K or N is a multiple of 64) skips
                        // the zero-filled second block.  wgrad: a last stage with a partial
                        // step serves only its whole 16-row steps; the partial one comes from
                        // the tail buffer below.
                        const bool tstep = tv != 0 && kb == t.nkb - 1;
                        const int nsteps = tstep ? (valid >> 4)
                                                 : (valid < kBK ? (valid + 15) >> 4 : kBK / 16);
                        // One base descriptor per operand and stage; step kk adds its byte offset
                        // / 16 to the address field (bits 0-13), which never carries out of it
                        // (shared memory is below 256 KB).  This thread issues every MMA of the
                        // pair, so its work per MMA bounds the mainloop: full stages run an
                        // unrolled loop of constant offsets.
                        const uint64_t a0 = (OP == OP_FWD) ? sdesc_sw128(a_addr, 16, 1024)
                                                           : sdesc_sw128(a_addr, kSubBytes, 1024);
                        const uint64_t b0 = (OP == OP_WGRAD) ? sdesc_sw128(b_addr, kSubBytes, 1024)
                                                             : sdesc_sw128(b_addr, 16, 1024);
                        const uint32_t acc0 = kb != kb0 ? 1u : 0u;
                        if (nsteps == kBK / 16) {
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk)
                                umma_bf16_pair(d_tmem, a0 + a_step<OP>(kk), b0 + b_step<OP>(kk, b_sub),
                                               idesc, kk ? 1u : acc0);
                        } else {
                            for (int kk = 0; kk < nsteps; ++kk)
                                umma_bf16_pair(d_tmem, a0 + a_step<OP>(kk), b0 + b_step<OP>(kk, b_sub),
                                               idesc, kk ? 1u : acc0);
                        }
                        umma_commit_pair(&c->empty[stage], 3);
                        if (++stage == R::kStages) { stage = 0; phase ^= 1u; }
                        if (tstep) {
                            const int tb = jt & 1;
                            if (!wait_bar(&c->tb_fixed[tb], (jt >> 1) & 1, c, pr, p.err)) { ok = false; break; }
                            tc_fence_after();
                            // G blocks and X blocks: 16 rows x 128 B each, the two 64-wide blocks
                            // of an operand kTailSub apart (LBO).
                            const uint32_t ta = smem_u32(tail_area + tb * kTailBytes);
                            umma_bf16_pair(d_tmem, sdesc_sw128(ta, kTailSub, 1024),
                                           sdesc_sw128(ta + 2 * kTailSub, kTailSub, 1024), idesc,
                                           (kb != kb0 || nsteps != 0) ? 1u : 0u);
                            umma_commit_pair(&c->tb_empty[tb], 3);
                            ++jt;
                        }
                    }
                    if (!ok) break;
                    // Arrives once this chunk's MMAs (if any: an empty group has none) are done.
                    umma_commit_pair(&c->tfull[A], 3);
                    acq.bump(A);
                }
                if (nch == 1) nextb ^= 1;
            }
            // Every MMA this thread issued has completed once this commit arrives.
            umma_commit_pair(&c->drain, 1);
            drain_wait(&c->drain, 0);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ---------------------------------------------------------- wgrad tail fixer (both CTAs)
        // Zeroes the rows past the unit's end in this CTA's copy of each tail step, then tells
        // the even CTA's MMA.
        if (OP == OP_WGRAD) {
            int jt = 0;
            Tile t;
            while (walker_next<OP, RT>(wk, p, sh, t)) {
                const int v = tail_rows(t.nred, t.nkb);
                if (!v) continue;
                const int tb = jt & 1;
                if (!wait_bar_warp(&c->tb_full[tb], (jt >> 1) & 1, c, pr, p.err)) break;
                // Rows [v % 16, 16) of the four 16-row blocks; lane l zeroes 16-byte chunk l % 8
                // of rows v % 16 + l / 8, + 4, ...  A whole 128-byte row is zeroed, so the
                // swizzle of its chunks does not matter.
                uint8_t* base = tail_area + tb * kTailBytes + (lane & 7) * 16;
#pragma unroll
                for (int bx = 0; bx < 4; ++bx)
                    for (int r = (v & 15) + (lane >> 3); r < 16; r += 4)
                        *reinterpret_cast<uint4*>(base + bx * kTailSub + r * 128) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (even) mbar_arrive(&c->tb_fixed[tb]);
                    else mbar_arrive_cluster(mapa_shared(smem_u32(&c->tb_fixed[tb]), 0u));
                }
                ++jt;
            }
        }
    } else if (warp >= 4 && OP == OP_WGRAD) {
        // ---------------------------------------------------------- wgrad epilogue (both CTAs)
        // Each warp writes 32 dW rows (its TMEM lanes) x 128 columns (one half of the tile) in
        // boxes of 32 rows x 64 bytes (32 bf16 or 16 fp32 columns): TMEM -> registers (one row
        // per thread) -> shared memory (64-byte swizzle) -> registers in line order (4 threads
        // per 64-byte row piece) -> coalesced global stores.  With accumulate the old
        // values are loaded in the same line order, a few boxes ahead, and added there.  (An
        // L2 prefetch of the unit's output block at the start of its mainloop was dropped:
        // the prefetched lines were often evicted before the epilogue read them, so the
        // wgrad-heavy accumulate read main_grad from HBM twice.)
        const int q = warp & 3, ew = warp - 4;          // TMEM lanes [32q, 32q + 32)
        const int hc = ew >> 2;                         // columns [128 hc, 128 hc + 128)
        const int mrow0 = kBM * static_cast<int>(pr.rank) + q * 32;   // first row of the pair tile
        const uint32_t tempty0 = mapa_shared(smem_u32(&c->tempty[0]), 0u);
        uint8_t* box = stage_area + ew * kEpiBoxBytes;
        constexpr bool acc = EPI == EPI_FP32_ACC || EPI == EPI_BF16_ACC;
        constexpr bool f32 =
            EPI == EPI_FP32 || EPI == EPI_FP32_ACC || EPI == EPI_PARTIAL || EPI == EPI_RED;
        constexpr int osz = f32 ? 4 : 2;
        const int rr = lane >> 2, gg = lane & 3;        // line-order phase: rows rr + 8j, chunk gg
        uint8_t* wslot = box + lane * 64;               // this lane's row in the write phase
        const int wsw = (lane >> 1) & 3;                // 64-byte swizzle: chunk g at g ^ wsw
        bool ok = true;
        int nextb = 0;
        Acq acq;                        // tfull phases waited for, per buffer
        Tile t;
        while (ok && walker_next<OP, RT>(wk, p, sh, t)) {
            const int nch = chunks_of<OP, EPI>(t.nkb);
            const int A = nextb, B = nextb ^ 1;
            const uint32_t lanebase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            const int cend = min(128 * hc + 128, t.ncols);
            uint8_t* obase;
            size_t ldo;
            if (EPI == EPI_PARTIAL) {
                obase = reinterpret_cast<uint8_t*>(p.partial) +
                        (static_cast<size_t>(t.u) * kPairM + mrow0) * kBN * 4;
                ldo = static_cast<size_t>(kBN) * 4;
            } else {
                ldo = static_cast<size_t>(p.ld_out) * osz;
                obase = reinterpret_cast<uint8_t*>(p.out) +
                        (static_cast<size_t>(t.e) * p.es_out +
                         static_cast<size_t>(t.f0 + mrow0) * p.ld_out + t.c0) * osz;
            }
            // This warp's (up to) 128 columns as boxes of 32 rows x 64 bytes (16 fp32 or 32
            // bf16 columns; up to 8 or 4 boxes).  Box b is bytes [64 b, 64 b + 64) of the
            // warp's row segments.  With accumulate, the old values of the next kAhead boxes
            // are always in flight.  A row past N or a 16-byte chunk past K (K % 8 == 0, so a
            // chunk is all in or all out) is neither read nor written; the split form's partial
            // tiles are written whole.
            constexpr int kBoxCols = f32 ? 16 : 32;
            constexpr int kBoxes = 128 / kBoxCols;
            constexpr int kAhead = acc ? 3 : 1;
            constexpr int kChunkCols = 16 / osz;
            const int nbox = (max(0, cend - 128 * hc) + kBoxCols - 1) / kBoxCols;
            const int nvalid = EPI == EPI_PARTIAL ? 32 : p.N - (t.f0 + mrow0);   // rows of the warp
            const int kvalid = EPI == EPI_PARTIAL ? 128 : p.K - (t.c0 + 128 * hc);
            auto inside = [&](int b, int j) {
                return rr + 8 * j < nvalid && b * kBoxCols + gg * kChunkCols < kvalid;
            };
            uint8_t* gseg = obase + static_cast<size_t>(rr) * ldo + (128 * hc) * osz + gg * 16;
            uint4 old[kAhead][4];
            auto first_loads = [&]() {
                if constexpr (acc) {
                    // The whole row segment of this thread's TMEM lane into L2 (up to 4 lines),
                    // before the unit's MMAs finish: the boxes past the first kAhead then find
                    // their old values in L2 instead of HBM.
                    if (lane < nvalid) {
                        const uint8_t* prow = obase + static_cast<size_t>(lane) * ldo + (128 * hc) * osz;
                        const int seg = min(128, kvalid) * osz;       // bytes of the row segment
                        for (int o = 0; o < seg; o += 128) prefetch_l2(prow + o);
                    }
#pragma unroll
                    for (int b = 0; b < kAhead; ++b)
                        if (b < nbox)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                old[b][j] = inside(b, j) ? *reinterpret_cast<const uint4*>(
                                                              gseg + b * 64 + 8 * j * ldo)
                                                        : make_uint4(0, 0, 0, 0);
                }
            };
            int fb = A;                 // the buffer that ends up holding the unit's value
            if (nch > 1) {
                // Chunked unit: B receives chunk 0, then B = RN(B + chunk c) for c = 1, 2, ...
                // No MMA writes B meanwhile, and this warp's own reads of B's previous use
                // completed (tcgen05.wait::ld) before these stores, so B needs no barrier.
                for (int ch = 0; ch < nch; ++ch) {
                    if (!wait_bar_warp(&c->tfull[A], acq.of(A) & 1u, c, pr, p.err)) { ok = false; break; }
                    tc_fence_after();
                    for (int cb = 128 * hc; cb < cend; cb += 32) {
                        uint32_t ra[32], rb[32];
                        tmem_ld_32x32b_x32(lanebase + static_cast<uint32_t>(A * kBN + cb), ra);
                        if (ch > 0) tmem_ld_32x32b_x32(lanebase + static_cast<uint32_t>(B * kBN + cb), rb);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            rb[j] = ch > 0 ? __float_as_uint(__fadd_rn(__uint_as_float(rb[j]),
                                                                      __uint_as_float(ra[j])))
                                           : ra[j];
                        tmem_st_32x32b_x32(lanebase + static_cast<uint32_t>(B * kBN + cb), rb);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (even) mbar_arrive(&c->tempty[A]);
                        else mbar_arrive_cluster_cta(tempty0 + A * 8u);   // chunk drained
                    }
                    acq.bump(A);
                }
                if (!ok) break;
                fb = B;
                first_loads();
            } else {
                first_loads();   // old values do not depend on this unit's MMAs
                if (!wait_bar_warp(&c->tfull[A], acq.of(A) & 1u, c, pr, p.err)) { ok = false; break; }
                tc_fence_after();
                acq.bump(A);
            }
            const uint32_t taddr = lanebase + static_cast<uint32_t>(fb * kBN + 128 * hc);
            uint32_t r[kBoxCols];       // one box's columns: TMEM is read box by box
#pragma unroll
            for (int b = 0; b < kBoxes; ++b) {
                if (b >= nbox) break;
                {
                    if (t.nkb > 0) {
                        if constexpr (f32) tmem_ld_32x32b_x16(taddr + b * kBoxCols, r);
                        else tmem_ld_32x32b_x32(taddr + b * kBoxCols, r);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < kBoxCols; ++j) r[j] = 0u;   // +0.0f: empty group
                    }
                    if (b + 1 >= nbox) {
                        // Every TMEM column of the unit is in registers: hand the buffer back
                        // to the MMA before the remaining stores.
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (even) mbar_arrive(&c->tempty[fb]);
                            else mbar_arrive_cluster_cta(tempty0 + fb * 8u);   // TMEM drained
                        }
                    }
                }
                // One row per thread, four 16-byte chunks.
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint4 v;
                    if constexpr (f32) {
                        const uint32_t* w = r + 4 * g;
                        v = make_uint4(w[0], w[1], w[2], w[3]);
                    } else {
                        const uint32_t* w = r + 8 * g;
                        v = make_uint4(pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                       pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                       pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                       pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
                    }
                    *reinterpret_cast<uint4*>(wslot + ((g ^ wsw) << 4)) = v;
                }
                __syncwarp();
                uint8_t* gline = gseg + b * 64;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = rr + 8 * j;
                    uint4 v = *reinterpret_cast<const uint4*>(box + row * 64 +
                                                              ((gg ^ ((row >> 1) & 3)) << 4));
                    if constexpr (acc) {
                        const uint4 o = old[b % kAhead][j];
                        if constexpr (f32) {
                            // out = RN32(out + dW): fp32 out.add_(dW)
                            v = make_uint4(__float_as_uint(__fadd_rn(__uint_as_float(o.x), __uint_as_float(v.x))),
                                           __float_as_uint(__fadd_rn(__uint_as_float(o.y), __uint_as_float(v.y))),
                                           __float_as_uint(__fadd_rn(__uint_as_float(o.z), __uint_as_float(v.z))),
                                           __float_as_uint(__fadd_rn(__uint_as_float(o.w), __uint_as_float(v.w))));
                        } else {
                            // out = bf16(float(out) + float(bf16(dW))): bf16 out.add_(dW)
                            v.x = pack_bf16x2(__fadd_rn(bf16_lo(o.x), bf16_lo(v.x)), __fadd_rn(bf16_hi(o.x), bf16_hi(v.x)));
                            v.y = pack_bf16x2(__fadd_rn(bf16_lo(o.y), bf16_lo(v.y)), __fadd_rn(bf16_hi(o.y), bf16_hi(v.y)));
                            v.z = pack_bf16x2(__fadd_rn(bf16_lo(o.z), bf16_lo(v.z)), __fadd_rn(bf16_hi(o.z), bf16_hi(v.z)));
                            v.w = pack_bf16x2(__fadd_rn(bf16_lo(o.w), bf16_lo(v.w)), __fadd_rn(bf16_hi(o.w), bf16_hi(v.w)));
                        }
                    }
                    if (inside(b, j)) {
                        if constexpr (EPI == EPI_RED) red_add_v4_f32(gline + 8 * j * ldo, v);
                        else *reinterpret_cast<uint4*>(gline + 8 * j * ldo) = v;
                    }
                }
                if constexpr (acc) {
                    if (b + kAhead < nbox)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            old[b % kAhead][j] = inside(b + kAhead, j)
                                                     ? *reinterpret_cast<const uint4*>(
                                                           gseg + (b + kAhead) * 64 + 8 * j * ldo)
                                                     : make_uint4(0, 0, 0, 0);
                }
                __syncwarp();   // the box is rewritten by the next box
            }
            if (nbox == 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (even) mbar_arrive(&c->tempty[fb]);
                    else mbar_arrive_cluster_cta(tempty0 + fb * 8u);   // nothing to drain
                }
            }
            if (nch == 1) nextb ^= 1;
        }
        (void)ok;
    } else if (warp >= 4) {
        // ---------------------------------------------------------- fwd / dgrad epilogue
        const int q = warp & 3;                 // TMEM lanes [32q, 32q + 32)
        const int hc = (warp - 4) >> 2;         // columns [128 hc, 128 hc + 128)
        const int mrow = kBM * static_cast<int>(pr.rank) + q * 32 + lane;   // row of the pair tile
        const uint32_t tempty0 = mapa_shared(smem_u32(&c->tempty[0]), 0u);
        Tile t;
        for (int it = 0; walker_next<OP, RT>(wk, p, sh, t); ++it) {
            const int buf = it & 1;
            if (!wait_bar_warp(&c->tfull[buf], (it >> 1) & 1, c, pr, p.err)) break;
            tc_fence_after();
            const int f = t.f0 + mrow;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(buf * kBN);
            const int nchunks = min((t.ncols + 31) >> 5, 4 * hc + 4);
            for (int ch = 4 * hc; ch < nchunks; ++ch) {
                uint32_t r[32];
                if (t.nkb > 0) {
                    tmem_ld_32x32b_x32(taddr + ch * 32, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;   // +0.0f
                }
                const int fdim = (OP == OP_FWD) ? p.N : p.K;
                if (f < fdim) {
                    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
                    const int jn = min(32, t.ncols - ch * 32);
                    const int64_t row = t.c0 + ch * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn)
                            out[(row + j) * p.ld_out + f] = __float2bfloat16_rn(__uint_as_float(r[j]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (even) mbar_arrive(&c->tempty[buf]);
                else mbar_arrive_cluster_cta(tempty0 + buf * 8u);   // TMEM drained
            }
        }
    }

    // Neither CTA leaves (or frees TMEM) while the other may still signal its barriers or
    // read its shared memory.
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ ordered reduce

struct ReduceParams {
    const int32_t* offs;
    const float* partial;
    void* out;
    int64_t rows;
    int E, N, K;
    int offs_kind;
    int epi;            // EPI_BF16 / EPI_FP32 / EPI_BF16_ACC / EPI_FP32_ACC
    int split_rows;
    int max_units;
    int64_t ld_out, es_out;   // out strides (elements)
};

struct ReduceSmem {
    int64_t warp_tot[kReduceThreads / 32];
    int total;
    int start[kMaxE];
    int size[kMaxE];
    int prefix[kMaxE + 1];
};

// dW[e][n][k] = p_0 + p_1 + ... + p_{S_e - 1} (fp32, left to right; +0.0 when S_e = 0),
// then the same epilogue as the unsplit kernel.  4 consecutive k per thread.
__global__ void __launch_bounds__(kReduceThreads) wgrad_reduce_kernel(const __grid_constant__ ReduceParams p) {
    __shared__ ReduceSmem sm;
    Shape sh;
    sh.kt = (p.K + kBN - 1) / kBN;
    sh.ft = ((p.N + kPairM - 1) / kPairM) * sh.kt;
    build_schedule<OP_WGRAD>(p.offs, p.offs_kind, p.rows, p.E, p.split_rows, p.max_units, sh,
                             sm.start, sm.size, sm.prefix, sm.warp_tot, &sm.total);
    const int64_t NK = static_cast<int64_t>(p.N) * p.K;
    const int64_t total4 = static_cast<int64_t>(p.E) * NK / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x; i < total4;
         i += static_cast<int64_t>(gridDim.x) * kReduceThreads) {
        const int64_t idx = i * 4;
        const int e = static_cast<int>(idx / NK);
        const int64_t rem = idx - e * NK;
        const int n = static_cast<int>(rem / p.K);
        const int k = static_cast<int>(rem - static_cast<int64_t>(n) * p.K);
        const int S = static_cast<int>((static_cast<int64_t>(sm.size[e]) + p.split_rows - 1) / p.split_rows);
        const int tile = (n / kPairM) * sh.kt + k / kBN;
        const size_t within = static_cast<size_t>(n % kPairM) * kBN + (k % kBN);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < S; ++s) {
            // prefix <= max_units and s * ft + tile < the group's own count <= max_units.
            const int64_t u = static_cast<int64_t>(sm.prefix[e]) + static_cast<int64_t>(s) * sh.ft + tile;
            if (u >= p.max_units) break;
            const float4 v = *reinterpret_cast<const float4*>(
                p.partial + static_cast<size_t>(u) * kPartialElems + within);
            if (s == 0) acc = v;
            else acc = make_float4(__fadd_rn(acc.x, v.x), __fadd_rn(acc.y, v.y),
                                   __fadd_rn(acc.z, v.z), __fadd_rn(acc.w, v.w));
        }
        // Four consecutive k of one row (K % 8 == 0): one 16-byte (fp32) or 8-byte (bf16) access.
        const int64_t off = static_cast<int64_t>(e) * p.es_out + static_cast<int64_t>(n) * p.ld_out + k;
        if (p.epi == EPI_FP32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + off) = acc;
        } else if (p.epi == EPI_FP32_ACC) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
            const float4 old = *o;
            *o = make_float4(__fadd_rn(old.x, acc.x), __fadd_rn(old.y, acc.y),
                             __fadd_rn(old.z, acc.z), __fadd_rn(old.w, acc.w));
        } else {
            uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + off);
            uint2 d;
            d.x = pack_bf16x2(acc.x, acc.y);
            d.y = pack_bf16x2(acc.z, acc.w);
            if (p.epi == EPI_BF16_ACC) {
                const uint2 old = *o;
                d.x = pack_bf16x2(__fadd_rn(bf16_lo(old.x), bf16_lo(d.x)),
                                  __fadd_rn(bf16_hi(old.x), bf16_hi(d.x)));
                d.y = pack_bf16x2(__fadd_rn(bf16_lo(old.y), bf16_lo(d.y)),
                                  __fadd_rn(bf16_hi(old.y), bf16_hi(d.y)));
            }
            *o = d;
        }
    }
}

// ------------------------------------------------------------------ non-deterministic split

struct DenseParams {
    void* out;              // [E][N][K] with strides ld_out, es_out (elements)
    const float* acc;       // finish: dense fp32 [E][N][K] sums
    int E, N, K;
    int epi;                // finish: EPI_BF16 or EPI_BF16_ACC
    int64_t ld_out, es_out;
};

// out[e][n][k] = +0.0f over a strided fp32 [E][N][K] (the destination of the unordered adds).
__global__ void __launch_bounds__(kReduceThreads) zero_f32_kernel(const __grid_constant__ DenseParams p) {
    const int64_t NK = static_cast<int64_t>(p.N) * p.K;
    const int64_t total4 = static_cast<int64_t>(p.E) * NK / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x; i < total4;
         i += static_cast<int64_t>(gridDim.x) * kReduceThreads) {
        const int64_t idx = i * 4;
        const int e = static_cast<int>(idx / NK);
        const int64_t rem = idx - e * NK;
        const int n = static_cast<int>(rem / p.K);
        const int k = static_cast<int>(rem - static_cast<int64_t>(n) * p.K);
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + e * p.es_out +
                                   static_cast<int64_t>(n) * p.ld_out + k) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// bf16 out from the fp32 sums: out = bf16(acc), or bf16(float(out) + float(bf16(acc))).
__global__ void __launch_bounds__(kReduceThreads) finish_bf16_kernel(const __grid_constant__ DenseParams p) {
    const int64_t NK = static_cast<int64_t>(p.N) * p.K;
    const int64_t total4 = static_cast<int64_t>(p.E) * NK / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x; i < total4;
         i += static_cast<int64_t>(gridDim.x) * kReduceThreads) {
        const int64_t idx = i * 4;
        const int e = static_cast<int>(idx / NK);
        const int64_t rem = idx - e * NK;
        const int n = static_cast<int>(rem / p.K);
        const int k = static_cast<int>(rem - static_cast<int64_t>(n) * p.K);
        const float4 a = *reinterpret_cast<const float4*>(p.acc + idx);
        uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + e * p.es_out +
                                            static_cast<int64_t>(n) * p.ld_out + k);
        uint2 d;
        d.x = pack_bf16x2(a.x, a.y);
        d.y = pack_bf16x2(a.z, a.w);
        if (p.epi == EPI_BF16_ACC) {
            const uint2 old = *o;
            d.x = pack_bf16x2(__fadd_rn(bf16_lo(old.x), bf16_lo(d.x)),
                              __fadd_rn(bf16_hi(old.x), bf16_hi(d.x)));
            d.y = pack_bf16x2(__fadd_rn(bf16_lo(old.y), bf16_lo(d.y)),
                              __fadd_rn(bf16_hi(old.y), bf16_hi(d.y)));
        }
        *o = d;
    }
}

}  // namespace gdg
