// sv_internal.h -- constants shared by the launch planner (planner.cpp) and the
// verify kernel (spec_verify.cu).  Not part of the public ABI.
#pragma once

#include <stdint.h>

namespace sv {

constexpr int kMaxK = 32;               // drafts per sequence
constexpr int kMaxRows = kMaxK + 1;     // target rows per sequence
constexpr int kMaxCluster = 16;         // CTAs per thread-block cluster (non-portable limit)
constexpr int kMinSlice = 1024;         // vocabulary entries per CTA before the planner shrinks the cluster
constexpr int kSliceAlign = 8;          // slices start on 8-entry boundaries (16 bytes of bf16)
constexpr int kRowBufAlign = 128;       // bytes; each staged row slice starts on this boundary
constexpr int kFixedSmem = 3072;        // bytes reserved for the kernel's fixed shared state

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Per-warp (max, sum) partials: [2 parities][group rows][warps] float pairs,
// then [2][warps] timeout flags.
inline int64_t partial_bytes(int group, int threads) {
    const int64_t nw = threads / 32;
    return 2 * group * nw * 8 + round_up(2 * nw * 4, 16);
}

// Shared-memory bytes a CTA needs for a plan: staged row slices, the fixed
// state, the partials, and one float per (tile, warp) for the draw.
inline int64_t smem_bytes_for(int64_t slice, int elem_bytes, int group, int threads) {
    const int E = 16 / elem_bytes;
    const int64_t rowbuf = round_up(slice * elem_bytes, kRowBufAlign);
    const int64_t tiles = ceil_div(ceil_div(slice, E), threads);
    return group * rowbuf + kFixedSmem + partial_bytes(group, threads) +
           tiles * (threads / 32) * 4 + kRowBufAlign;
}

}  // namespace sv
