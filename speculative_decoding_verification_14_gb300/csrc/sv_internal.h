// sv_internal.h -- constants and shared-memory layout shared by the launch
// planner (planner.cpp) and the verify kernel (spec_verify.cu).  Not part of
// the public ABI.
#pragma once

#include <stdint.h>

namespace sv {

constexpr int kMaxK = 32;               // drafts per sequence
constexpr int kMaxRows = kMaxK + 1;     // target rows per sequence
constexpr int kMaxCluster = 16;         // CTAs per thread-block cluster (non-portable limit)
constexpr int kSliceAlign = 8;          // slices start on 8-entry boundaries (16 bytes of bf16)
constexpr int kStages = 3;              // ring stages per warp (batches that fill the GPU)
// Batches whose clusters leave SMs room take deeper rings: kStagesDeep
// stages per warp, kDeepCtasPerSM 128-thread CTAs per SM (the launch bounds
// of those kernels), so a warp keeps more of its stretch in flight.
constexpr int kStagesDeep = 6;
constexpr int kDeepCtasPerSM = 4;
// Wait limits (fixed; nothing at run time shortens them).  A wait on another
// CTA's or warp's progress (pushed partials, a posted decision) gives up after
// kWaitNs and the sequence reports SV_ERR_TIMEOUT.  A wait on one of the
// warp's own global-to-shared bulk copies depends on no other CTA and always
// ends; it has a limit of its own, kCopyWaitNs.
constexpr unsigned long long kWaitNs = 2000000000ull;       // 2 s
constexpr unsigned long long kCopyWaitNs = 10000000000ull;  // 10 s
constexpr int kChunkBytes = 2048;       // bytes per ring stage (one bulk copy)
constexpr int kDrawTile = kChunkBytes / 4;  // entries per draw tile (its draft row fills one stage)
constexpr int kFixedSmem = 3072;        // bytes reserved for the kernel's fixed shared state
constexpr int kSmemPerSM = 233472;      // shared memory of one SM (228 KB)
constexpr int kSmemPerCtaReserved = 1024;  // the runtime's per-CTA reservation
constexpr int kSmemOptinPerCta = 232448;   // shared memory one CTA may opt into (227 KB)
constexpr int kThreadsPerSM = 896;      // resident threads the kernels' launch bounds target (7 CTAs of 128)

constexpr int kGreedyDepth = 8;         // greedy kernel: 16-byte loads in flight per lane
constexpr int kGreedyCtasPerSM = 8;     // greedy kernel: resident 128-thread CTAs per SM (launch bounds)
constexpr int kTruncCtasPerSM = 4;      // truncated-target kernel: resident CTAs per SM (launch bounds)
constexpr int kTruncMaxCluster = 8;     // truncated-target kernel: largest cluster (shared histograms)

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Shared memory of one CTA: per-warp rings, the fixed state, the barriers
// (per-warp ring stages, then four exchange barriers: row partials of the two
// parities, draw totals of the two draw rounds), the row partials pushed by
// every warp of the cluster (offset, sum hi, sum lo, max: 16 bytes)
// [2 parities][group rows][cluster CTAs x warps], and the draw's per-warp tile
// totals with the offsets the bonus row's totals are taken against.
struct Layout {
    int64_t wvec;       // 16-byte vectors per warp stretch
    int64_t ntw;        // draw tiles (kDrawTile entries) per warp stretch
    int64_t off_fixed, off_bar, off_part, off_tt, total;
};

constexpr int kExchangeBarriers = 4;

inline Layout layout_for(int64_t slice, int elem_bytes, int group, int threads, int cluster,
                         int stages = kStages) {
    const int64_t nw = threads / 32;
    const int64_t E = 16 / elem_bytes;
    Layout l;
    l.wvec = ceil_div(ceil_div(slice, E), nw);
    l.ntw = ceil_div(l.wvec * E, kDrawTile);
    l.off_fixed = nw * stages * kChunkBytes;
    l.off_bar = l.off_fixed + kFixedSmem;
    l.off_part = l.off_bar + round_up((nw * stages + kExchangeBarriers) * 8, 16);
    l.off_tt = l.off_part + round_up(2 * (int64_t)group * cluster * nw * 16, 16);
    l.total = l.off_tt + round_up(2 * nw * l.ntw * 4, 16);  // tile totals, then their offsets
    return l;
}

// Greedy verification kernel (greedy.cu): launch description and entry points.
struct GreedyLaunch {
    const void* logits;
    const int32_t* tokens;
    int32_t* accept_len;
    int32_t* out_tokens;
    uint8_t* accept_mask;
    int32_t* row_argmax;
    int32_t* status;
    uint32_t* err_word;
    uint32_t* al_hist;
    int64_t V, slice;
    int B, K, C;
    int es;   // bytes per logit (2 or 4)
    int vec;  // 1: 16-byte vector loads (aligned rows)
    unsigned long long wait_ns;  // give up on a row's partials after this long
};
int greedy_set_attributes();                              // 0 on success
int greedy_launch(const GreedyLaunch& g, void* stream);  // 0 on success

// Truncated-target verification kernel (truncated.cu).
struct TruncLaunch {
    const void* logits;
    const float* q;
    const int32_t* tokens;
    const float* u;
    int32_t* accept_len;
    int32_t* out_tokens;
    uint8_t* accept_mask;
    float* row_stats;
    float* p_draft;
    int32_t* status;
    uint32_t* err_word;
    uint32_t* al_hist;
    int64_t V, slice;
    int B, K, C;
    int es, vec, qvec;
    float c, T, dmin;
    double top_p;
    unsigned long long wait_ns;
    const void* dlogits;  // draft logits [B, K, V] in the target's dtype (q unused), or NULL
    float cd;             // log2(e) / T_draft rounded to float (draft logits)
};
int trunc_launch(const TruncLaunch& g, void* stream);    // 0 on success

}  // namespace sv
