// vcd_plan.h -- how the [S, C] token x channel plane is cut into work units.
//
// A lane owns VEC consecutive channels (2 * VEC bytes of BF16 per token, 4
// channels in both directions); a warp owns 32 lanes, i.e. one row segment of
// 32 * VEC channels per token; a "column" is those channels, a "row" a run of
// L consecutive tokens, and a unit is one (row, column) pair, processed by one
// warp token by token with a 3-token halo on the left (and on the right in the
// backward).
//
// The cut is a function of (S, C), the backward's launch shape and
// compile-time constants only -- never of the device -- so the backward's
// partial rows, and therefore its fixed-order reduction, are the same on every
// GPU: gradients are bitwise reproducible per (S, C, route), where the route
// (weight / bias dtypes, SiLU' policy, launch shape) is chosen on the host from
// the call's arguments. The unit counts are sized so that one wave of the
// persistent grid takes every unit on GB300 (152 SMs x the kernel's resident
// warps per SM).
#pragma once
#include <stdint.h>

namespace vcd {

constexpr int kWarpsPerCta = 8;
constexpr int kThreadsPerCta = 32 * kWarpsPerCta;
#ifndef VCD_BWD_VEC
#define VCD_BWD_VEC 4
#endif
constexpr int kFwdVec = 4;                    // channels per lane, forward
constexpr int kBwdVec = VCD_BWD_VEC;          // channels per lane, backward
// The shortest unit a plan cuts: it binds only where S is small against the
// resident warps (fewer than 16 tokens per warp), where the time is latency
// and the parallelism counts for more than the 3-token halo's extra reads
// (4096 x 256: forward 16 -> 10 us, backward 30 -> 21 us against 64-token
// units, measured).
constexpr int64_t kMinTokensPerUnit = 16;
constexpr int kPartialStride = 5;             // dweight[0..3], dbias per channel

#ifndef VCD_FWD_CTAS_PER_SM
#define VCD_FWD_CTAS_PER_SM 3
#endif
constexpr int kFwdCtasPerSm = VCD_FWD_CTAS_PER_SM;
constexpr int64_t kGb300Sms = 152;
constexpr int64_t kFwdTargetUnits = kGb300Sms * kFwdCtasPerSm * kWarpsPerCta;

// Forward batch shapes: the same units and grid, different batches. Streaming
// takes 4-token batches in a 6-stage ring; short documents (a start in most
// batches, so each batch walks cu_seqlens and takes the masked path) take
// 16-token batches in a 2-stage ring, which quarters those per-batch costs.
// The choice changes no result, only the time.
// kFwdExact is the exactness-guarded route (conv1d_fwd_exact): 8-token
// batches on every workload, each element checked and the doubtful ones
// recomputed (vcd_fwd.cu).
enum FwdShape { kFwdStream = 0, kFwdShortDocs = 1, kFwdExact = 2 };

// Backward launch shapes: one CTA per SM either way; they trade registers for
// warps.
//   kBwdWide: 12 warps, up to 168 registers a thread -- mask-free streaming
//             whose 16-warp build would spill;
//   kBwdDeep: 16 warps, up to 128 registers a thread -- more warps to hide
//             latency, for the mask-free routes without a bias.
// bwd_shape() picks one per call.
//   kBwdChunked: 12 warps, up to 168 registers, 8-token batches and room in
//             shared memory for compensated per-chunk sums -- the "fp32"
//             policy's chunks of units of at most 256 tokens, and short
//             documents (masked paths) under either policy.
enum BwdShape { kBwdWide = 0, kBwdDeep = 1, kBwdChunked = 2 };
constexpr int kBwdShapeWarps[3] = {12, 16, 12};

// Mean document length (tokens) below which most batches hold a document
// start and take the masked path.
constexpr int64_t kShortDocTokens = 32;

// The forward's batch shape for a call.
inline int fwd_shape(int64_t S, int64_t num_docs) {
    return num_docs * kShortDocTokens >= S ? kFwdShortDocs : kFwdStream;
}

// The backward's launch shape for a call: chunked for the "fp32" policy (its
// short units need the shared-memory chunk sums) and for short documents
// (the masked interior path without the deep shape's spills: 131072 x 1032
// 174.7 -> 172.7 us, measured); under the "bf16" policy on longer documents
// deep for routes without a bias (those kernels keep all their state within
// 128 registers), wide with a bias, whose 16-warp kernels would spill. A
// function of the call's arguments only, so a route's partial rows are the
// same on every call and every device.
inline int bwd_shape(int64_t S, int64_t num_docs, int policy, bool has_bias) {
    if (policy == 1 || num_docs * kShortDocTokens >= S) return kBwdChunked;
    return has_bias ? kBwdWide : kBwdDeep;
}

struct Plan {
    int64_t S, C;
    int64_t col_channels;   // 32 * VEC
    int64_t groups;   // C / VEC
    int64_t ncols;    // columns of 32 groups (the last may be partial)
    int64_t rows;     // token ranges per column
    int64_t L;        // tokens per range (the last range may be shorter)
    int64_t units;    // ncols * rows
};

// The backward's plan adds its chunks: consecutive units of one column that
// one warp streams without restarting, each chunk one partial row. (Kept out
// of Plan: the forward's kernel arguments stay as small as they were, which
// its schedule was measured to depend on.)
struct BwdPlan : Plan {
    int64_t per;      // units per chunk
    int64_t chunks;   // chunks per column
    // The transposed narrow column (below); nfull == ncols and nnarrow == 0
    // when the last column runs like the others.
    int64_t nfull;    // columns in the normal mapping: chunk c of column k is assignment c nfull + k
    int64_t ng;       // four-channel groups of the transposed column
    int64_t h;        // pieces per chunk of the transposed column
    int64_t q;        // its chunks per warp
    int64_t nnarrow;  // its warps: assignments nfull chunks .. + nnarrow - 1
};

inline Plan make_plan(int64_t S, int64_t C, int vec, int64_t target_units) {
    Plan p;
    p.S = S;
    p.C = C;
    p.col_channels = 32 * vec;
    p.groups = C / vec;
    p.ncols = (p.groups + 31) / 32;
    int64_t rows = target_units / p.ncols;
    const int64_t cap = (S + kMinTokensPerUnit - 1) / kMinTokensPerUnit;
    if (rows > cap) rows = cap;
    if (rows < 1) rows = 1;
    p.L = S > 0 ? (S + rows - 1) / rows : 1;
    p.rows = S > 0 ? (S + p.L - 1) / p.L : 0;
    p.units = p.ncols * p.rows;
    return p;
}

inline Plan fwd_plan(int64_t S, int64_t C) { return make_plan(S, C, kFwdVec, kFwdTargetUnits); }

// The "fp32" SiLU' policy keeps each unit's FP32 dweight / dbias sums short
// (at most kFp32TokensPerUnit tokens, relative rounding error about
// 0.2 * 2^-24 * sqrt(256) = 2e-7); a warp streams a chunk of consecutive
// units of one column and adds each unit's sums into a compensated two-float
// accumulator, so the chunk's one partial row is its sum rounded once to
// FP32. The "bf16" policy's 5e-5 tolerance allows long units (one per chunk).
// Chunks are cut from GB300's resident warps per column (constants, not the
// device at hand), so the partial rows and their reduction order are the same
// on every device.
#ifndef VCD_FP32_UNIT_TOKENS
#define VCD_FP32_UNIT_TOKENS 256
#endif
constexpr int64_t kFp32TokensPerUnit = VCD_FP32_UNIT_TOKENS;

// The chunk is sized first (units per chunk: the fewest that let each column's
// warps cover S with units of at most kFp32TokensPerUnit tokens), then the
// unit is the shortest multiple of kFp32UnitAlign tokens that lets the
// column's chunks cover S: so each column gets close to its share of the
// resident warps (a fixed 256-token unit left 15% of them idle at S = 131072
// over 9 columns). Every unit but a column's last is L tokens long, L a
// multiple of the chunked shape's batch so that unit boundaries fall at the
// same position of a batch.
constexpr int64_t kFp32UnitAlign = 8;
static_assert(kFp32TokensPerUnit % kFp32UnitAlign == 0, "unit length must align");

// The narrow last column. When C's last 128-channel column holds g <= 16 of
// its 32 four-channel groups, a warp on it in the normal mapping costs as
// much per token as on a full column for g/32 of the data (C = 1032: 1/9 of
// the warp time for 1/129 of the elements). The backward transposes that
// column: a warp covers m = 32/g stretches ("pieces") of its tokens at once,
// g lanes on each, one per group. A chunk of the column is cut into h equal
// pieces (below), a warp takes q = m/h whole chunks and adds each chunk's
// pieces in piece order into the chunk's partial row. Those few warps take
// the whole column, and the full columns share the rest of the resident
// warps. The partial rows keep their layout (chunks x ncols rows); a
// transposed plan is capped at kMaxPartialRows of them. (The forward keeps
// the normal mapping: a transposed forward measured slower, its lanes'
// scattered 8-byte loads and stores costing more than the idle lanes.)
constexpr int64_t kNarrowMaxGroups = 16;
constexpr int64_t kMaxPartialRows = 3072;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The transposed plan for the last column's g groups, or false (p untouched)
// where none applies.
inline bool narrow_plan(BwdPlan& p, int64_t S, int64_t warps, int policy, int64_t g) {
    const int64_t m = 32 / g, nfull = p.ncols - 1;
    const int64_t row_cap = kMaxPartialRows / p.ncols;          // chunks per column at most
    const int64_t tok_cap = ceil_div(S, kMinTokensPerUnit);
    if (row_cap < 1) return false;
    // chunks per column W with W nfull + W / qq <= warps
    auto share = [&](int64_t qq) {
        const int64_t w = warps * qq / (nfull * qq + 1);
        return w < 1 ? 1 : w > row_cap ? row_cap : w;
    };
    // pieces per chunk: the smallest multiple of the chunk's units that is at
    // least 4 under the "bf16" policy, 6 under "fp32" (a transposed lane
    // takes about four times a full column lane's time per token, more with
    // the accurate SiLU'; measured), else the largest multiple that fits m
    const int64_t h_min = policy == 1 ? 6 : 4;
    auto pieces = [&](int64_t per) -> int64_t {
        int64_t h = (h_min + per - 1) / per * per;
        while (h > m && h > per) h -= per;
        return h;
    };
    // the plan for a target of wpc chunks per column
    auto make = [&](int64_t wpc, BwdPlan& r) -> bool {
        r = p;
        r.per = policy == 1 ? ceil_div(S, wpc * kFp32TokensPerUnit) : 1;
        const int64_t h = pieces(r.per);
        if (m / h < 1) return false;
        if (r.per > 1) {
            r.L = ceil_div(ceil_div(S, wpc * r.per), kFp32UnitAlign) * kFp32UnitAlign;
            r.rows = ceil_div(S, r.L);
            r.chunks = ceil_div(r.rows, r.per);
        } else {
            const int64_t rows = wpc < tok_cap ? wpc : tok_cap;
            r.L = ceil_div(S, rows);
            r.rows = ceil_div(S, r.L);
            r.chunks = r.rows;
        }
        r.units = r.ncols * r.rows;
        r.nfull = nfull;
        r.ng = g;
        r.h = h;
        r.q = m / h;
        r.nnarrow = ceil_div(r.chunks, r.q);
        return true;
    };
    // the most chunks per column whose assignments fit the resident warps,
    // from the estimate down
    BwdPlan r;
    int64_t wpc = share(m / pieces(1));
    for (;; --wpc) {
        if (!make(wpc, r)) return false;
        if (r.nfull * r.chunks + r.nnarrow <= warps || wpc == 1) break;
    }
    p = r;
    return true;
}

// transpose: allow the transposed narrow column (the exactness-guarded route
// keeps the normal mapping).
inline BwdPlan bwd_plan(int64_t S, int64_t C, int policy, int shape, bool transpose = true) {
    const int64_t warps = kGb300Sms * kBwdShapeWarps[shape];
    BwdPlan p;
    static_cast<Plan&>(p) = make_plan(S, C, kBwdVec, warps);
    p.per = 1;
    p.chunks = p.rows;
    p.nfull = p.ncols;
    p.ng = 0;
    p.h = 1;
    p.q = 0;
    p.nnarrow = 0;
    const int64_t g = p.groups - 32 * (p.ncols - 1);             // groups of the last column
    if (transpose && S > 0 && g <= kNarrowMaxGroups && narrow_plan(p, S, warps, policy, g)) return p;
    if (policy == 1 && p.L > kFp32TokensPerUnit && S > 0) {
        const int64_t wpc = warps / p.ncols > 0 ? warps / p.ncols : 1;   // warps per column
        p.per = (S + wpc * kFp32TokensPerUnit - 1) / (wpc * kFp32TokensPerUnit);
        const int64_t span = wpc * p.per;                                  // units per column at most
        p.L = (S + span - 1) / span;
        p.L = (p.L + kFp32UnitAlign - 1) / kFp32UnitAlign * kFp32UnitAlign;
        p.rows = (S + p.L - 1) / p.L;
        p.units = p.ncols * p.rows;
        p.chunks = (p.rows + p.per - 1) / p.per;
    }
    return p;
}

// Bytes of one route's partial rows: one FP32 row of 32 * kBwdVec channels x
// 5 values per chunk of each column.
inline uint64_t bwd_workspace_bytes_for(int64_t S, int64_t C, int policy, int shape,
                                        bool transpose = true) {
    if (S <= 0) return 0;
    const BwdPlan p = bwd_plan(S, C, policy, shape, transpose);
    return (uint64_t)p.chunks * p.ncols * p.col_channels * kPartialStride * sizeof(float);
}

// The most a policy's routes need over every call shape: the "fp32" policy
// always runs the chunked shape, the "bf16" policy the wide or the deep one.
inline uint64_t bwd_workspace_bytes_for(int64_t S, int64_t C, int policy) {
    if (policy == 1) return bwd_workspace_bytes_for(S, C, policy, kBwdChunked);
    const uint64_t d = bwd_workspace_bytes_for(S, C, policy, kBwdDeep);
    const uint64_t w = bwd_workspace_bytes_for(S, C, policy, kBwdWide);
    const uint64_t c = bwd_workspace_bytes_for(S, C, policy, kBwdChunked);
    const uint64_t m = w > d ? w : d;
    return c > m ? c : m;
}

// What one call needs.
inline uint64_t bwd_call_workspace_bytes(int64_t S, int64_t C, int64_t num_docs, int policy,
                                         bool has_bias) {
    return bwd_workspace_bytes_for(S, C, policy, bwd_shape(S, num_docs, policy, has_bias));
}

// The exactness-guarded backward (conv1d_bwd_exact) runs the chunked shape
// for both policies and adds, per chunk, a list of dx elements to recompute:
// room for one in 64 of the chunk's elements (at least 64; a few in 10^3 are
// listed on normal inputs), 8 bytes each, then one 4-byte count per chunk.
// The layout after the partial rows, each part starting on a 16-byte boundary.
inline int64_t exact_list_cap(const BwdPlan& p) {
    const int64_t elems = p.L * p.per * p.col_channels;
    const int64_t cap = elems / 64;
    return cap > 64 ? cap : 64;
}
inline uint64_t round16(uint64_t n) { return (n + 15) & ~(uint64_t)15; }
struct ExactLayout {
    uint64_t partial_bytes, list_offset, count_offset, total;
    int64_t cap;
};
inline ExactLayout exact_layout(int64_t S, int64_t C, int policy) {
    ExactLayout e = {0, 0, 0, 0, 0};
    if (S <= 0) return e;
    const BwdPlan p = bwd_plan(S, C, policy, kBwdChunked, false);
    const uint64_t lists = (uint64_t)p.chunks * p.ncols;
    e.cap = exact_list_cap(p);
    e.partial_bytes = round16(bwd_workspace_bytes_for(S, C, policy, kBwdChunked, false));
    e.list_offset = e.partial_bytes;
    e.count_offset = round16(e.list_offset + lists * (uint64_t)e.cap * 8);
    e.total = round16(e.count_offset + lists * 4);
    return e;
}
inline uint64_t bwd_exact_workspace_bytes(int64_t S, int64_t C) {
    const uint64_t a = exact_layout(S, C, 0).total, b = exact_layout(S, C, 1).total;
    return a > b ? a : b;
}

// The most any route needs.
inline uint64_t bwd_workspace_bytes(int64_t S, int64_t C) {
    const uint64_t a = bwd_workspace_bytes_for(S, C, 0), b = bwd_workspace_bytes_for(S, C, 1);
    return a > b ? a : b;
}

}  // namespace vcd
