// vcd_plan.h -- how the [S, C] token x channel plane is cut into work units.
//
// A lane owns VEC consecutive channels (one 16-byte BF16 vector for VEC = 8,
// 8 bytes for VEC = 4); a warp owns 32 such groups of one token range, so
// each warp-wide load is one contiguous row segment. A "column" is the 32 * VEC
// channels of one warp, a "row" a run of L consecutive tokens; a unit is one
// (row, column) pair and is processed by one warp, token by token, with a
// 3-token halo on the left (and on the right in the backward).
//
// The cut is a function of (S, C) and compile-time constants only -- never of
// the device -- so the backward's partial rows, and therefore its fixed-order
// reduction, are the same on every GPU: gradients are bitwise reproducible
// per (S, C, route). The unit count is sized so that one wave of the
// persistent grid (152 SMs x 16 resident warps on GB300) takes every unit.
#pragma once
#include <stdint.h>

namespace vcd {

constexpr int kWarpsPerCta = 8;
constexpr int kThreadsPerCta = 32 * kWarpsPerCta;
constexpr int64_t kTargetUnits = 152 * 16;   // GB300: 152 SMs x 16 warps
constexpr int64_t kMinTokensPerUnit = 64;    // keeps the 3-token halo below 5%
#ifndef VCD_FWD_VEC
#define VCD_FWD_VEC 8
#endif
constexpr int kFwdVec = VCD_FWD_VEC;      // channels per lane, forward
constexpr int kBwdVec = 4;                // channels per lane, backward
constexpr int kPartialStride = 5;            // dweight[0..3], dbias per channel

struct Plan {
    int64_t S, C;
    int64_t groups;   // C / vec
    int64_t ncols;    // columns of 32 groups (the last may be partial)
    int64_t rows;     // token ranges per column
    int64_t L;        // tokens per range (the last range may be shorter)
    int64_t units;    // ncols * rows
};

inline Plan make_plan(int64_t S, int64_t C, int vec) {
    Plan p;
    p.S = S;
    p.C = C;
    p.groups = C / vec;
    p.ncols = (p.groups + 31) / 32;
    int64_t rows = kTargetUnits / p.ncols;
    int64_t cap = (S + kMinTokensPerUnit - 1) / kMinTokensPerUnit;
    if (rows > cap) rows = cap;
    if (rows < 1) rows = 1;
    p.L = S > 0 ? (S + rows - 1) / rows : 1;
    p.rows = S > 0 ? (S + p.L - 1) / p.L : 0;
    p.units = p.ncols * p.rows;
    return p;
}

// Bytes of the backward's partial rows: one FP32 row of 32 * kBwdVec channels
// x 5 values per unit.
inline uint64_t bwd_workspace_bytes(int64_t S, int64_t C) {
    if (S <= 0) return 0;
    Plan p = make_plan(S, C, kBwdVec);
    return (uint64_t)p.units * 32 * kBwdVec * kPartialStride * sizeof(float);
}

}  // namespace vcd
