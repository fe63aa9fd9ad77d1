// planner.cpp -- maps one batched verify onto thread-block clusters.
//
// Work unit: one sequence b (its K+1 target rows, K draft rows, K tokens and
// K+1 uniforms) is verified by one cluster of C CTAs.  CTA r owns the
// vocabulary slice [r*slice, (r+1)*slice) of every row of b and each warp a
// contiguous stretch of that slice, streamed through a small private ring of
// shared memory; the partial softmax statistics of a row meet inside the
// cluster through distributed shared memory.
//
// Choice of C: the sequences' rows are consumed one after another (the test
// loop of [P1] stops at the first rejection, so later rows are not read), so
// a sequence is a chain of dependent steps and throughput comes from running
// many sequences at once.  The planner takes the largest cluster that still
// lets every sequence of the batch be resident at the same time (more CTAs per
// sequence shorten each step), while keeping at least half a ring stage of
// work per warp; batches too large to be resident get C = 1.
//
// Rows per step (group): 1 when the batch fills the GPU (only rows the loop
// reaches are read; the first chunks of the next row are prefetched while a
// row is decided); all K+1 for batches too small to fill it, where latency
// rules and one barrier decides every row.
//
// Ring depth: three 2 KB stages per warp, or six when the plan's CTAs fit at
// four per SM with the deeper rings (batches that leave SMs room).
//
// [P1] = reactapp.top, "Speculative decoding and early exit: speeding up
// autoregressive decode", section "Speculative decoding: draft first, then
// verify".
#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace {

// dl: verification with draft logits -- every test row's draft row streams
// with it, so each group row holds two rows of partials; 128 threads only.
int plan_impl(int num_sms, int smem_per_cta, int max_cluster, int B, int K, int64_t V, int dtype,
              int ovr_cluster, int ovr_group, int ovr_threads, sv_plan* out, bool dl = false) {
    using namespace sv;
    if (!out || num_sms < 1 || smem_per_cta < 1 || max_cluster < 1 || B < 1 || K < 0 ||
        K > kMaxK || V < 1 || V > ((int64_t)1 << 31) || (dtype != SV_F32 && dtype != SV_BF16))
        return SV_ERR_INVALID_ARG;
    if (ovr_cluster < 0 || ovr_cluster > kMaxCluster || ovr_group < 0 ||
        (ovr_threads != 0 && ovr_threads != 128 && ovr_threads != 256 && ovr_threads != 512))
        return SV_ERR_INVALID_ARG;
    if (ovr_cluster > max_cluster)
        return SV_ERR_UNSUPPORTED;
    const int es = dtype == SV_BF16 ? 2 : 4;
    const int E = 16 / es;
    const int rows = K + 1;
    if (dl && ovr_threads != 0 && ovr_threads != 128)
        return SV_ERR_INVALID_ARG;
    const int threads = ovr_threads ? ovr_threads : 128;
    const int pr = dl ? 2 : 1;  // partial rows per group row
    const int nw = threads / 32;
    const int cmax = max_cluster < kMaxCluster ? max_cluster : kMaxCluster;
    const int64_t min_slice = (int64_t)nw * (kChunkBytes / 16) * E / 2;  // half a stage per warp
    // when the batch fills the GPU, each warp keeps at least 4 ring stages of
    // work per row: below that the per-row partial, barrier and merge cost more
    // than the streaming they serve
    const int64_t min_slice_full = (int64_t)nw * 4 * (kChunkBytes / 16) * E;

    // resident CTAs per SM with a single-row plan (threads and shared memory)
    const int64_t smem1 = layout_for(round_up(ceil_div(V, 4), kSliceAlign), es, pr, threads, 4).total;
    int64_t per_sm = (int64_t)kSmemPerSM / (smem1 + kSmemPerCtaReserved);
    const int64_t by_threads = kThreadsPerSM / threads;  // the kernels' launch bounds
    if (per_sm > by_threads)
        per_sm = by_threads;
    if (per_sm < 1)
        per_sm = 1;
    const int64_t capacity = per_sm * num_sms;

    int C;
    if (ovr_cluster) {
        C = ovr_cluster;
    } else {
        C = 1;
        for (int c = cmax >= 16 ? 16 : cmax; c >= 1; c /= 2) {
            const bool fills = (int64_t)B * c >= num_sms;
            if ((int64_t)B * c <= capacity &&
                (c == 1 || ceil_div(V, c) >= (fills ? min_slice_full : min_slice))) {
                C = c;
                break;
            }
        }
    }
    int G;
    if (ovr_group)
        G = ovr_group < rows ? ovr_group : rows;
    else
        G = (int64_t)B * C >= num_sms ? 1 : rows;

    const int64_t slice = round_up(ceil_div(V, C), kSliceAlign);
    Layout l = layout_for(slice, es, pr * G, threads, C);
    while (l.total > smem_per_cta && G > 1 && !ovr_group) {
        G = (G + 1) / 2;
        l = layout_for(slice, es, pr * G, threads, C);
    }
    if (l.total > smem_per_cta)
        return SV_ERR_UNSUPPORTED;
    // Deeper rings when the plan's CTAs are few enough to be resident at the
    // deep kernels' occupancy: a warp then keeps more of its stretch in flight,
    // which shortens every step of a latency-bound chain.
    int stages = kStages;
    if (threads == 128) {
        const Layout ld = layout_for(slice, es, pr * G, threads, C, kStagesDeep);
        int64_t per_sm_deep = (int64_t)kSmemPerSM / (ld.total + kSmemPerCtaReserved);
        if (per_sm_deep > kDeepCtasPerSM)
            per_sm_deep = kDeepCtasPerSM;
        if (ld.total <= smem_per_cta && (int64_t)B * C <= per_sm_deep * num_sms) {
            stages = kStagesDeep;
            l = ld;
        }
    }
    out->cluster = C;
    out->group = G;
    out->threads = threads;
    out->smem_bytes = (int)l.total;
    out->slice = slice;
    out->grid = (int64_t)B * C;
    out->bulk_copy = ((V * es) % 16) == 0 ? 1 : 0;
    out->prefetch_next = G == 1 ? 1 : 0;
    out->stages = stages;
    return SV_OK;
}

}  // namespace

extern "C" int spec_verify_plan_for(int num_sms, int smem_per_cta, int max_cluster, int B, int K,
                                    int64_t V, int logits_dtype, int ovr_cluster, int ovr_group,
                                    int ovr_threads, sv_plan* out) {
    return plan_impl(num_sms, smem_per_cta, max_cluster, B, K, V, logits_dtype, ovr_cluster,
                     ovr_group, ovr_threads, out);
}

// Greedy verification (greedy.cu): the same mapping -- one cluster of C CTAs
// per sequence, vocabulary slices, rows in order -- with no shared-memory
// ring, so residency is set by the kernel's launch bounds (eight 128-thread
// CTAs per SM).  Each lane keeps eight 16-byte loads in flight; a batch that
// fills the GPU gets at least two such rounds per warp and row, a smaller
// batch the largest cluster that leaves every lane one vector.
namespace {

// Cluster-per-sequence plan for the kernels without a shared-memory ring
// (greedy and truncated-target verification): ctas_per_sm resident 128-thread
// CTAs per SM, `depth` 16-byte loads in flight per lane, clusters up to cap.
int plan_rows(int num_sms, int max_cluster, int B, int K, int64_t V, int logits_dtype,
              int ovr_cluster, int ctas_per_sm, int depth, int cap, sv_plan* out) {
    using namespace sv;
    if (!out || num_sms < 1 || max_cluster < 1 || B < 1 || K < 0 || K > kMaxK || V < 1 ||
        V > ((int64_t)1 << 31) || (logits_dtype != SV_F32 && logits_dtype != SV_BF16) ||
        ovr_cluster < 0 || ovr_cluster > cap)
        return SV_ERR_INVALID_ARG;
    if (ovr_cluster > max_cluster)
        return SV_ERR_UNSUPPORTED;
    const int es = logits_dtype == SV_BF16 ? 2 : 4;
    const int64_t E = 16 / es;
    const int nw = 4;
    const int64_t capacity = (int64_t)ctas_per_sm * num_sms;
    const int64_t min_full = (int64_t)nw * 32 * depth * E * 2;
    const int64_t min_small = (int64_t)nw * 32 * E;
    const int cmax = max_cluster < cap ? max_cluster : cap;
    int C = 1;
    if (ovr_cluster) {
        C = ovr_cluster;
    } else {
        for (int c = cmax >= 16 ? 16 : cmax; c >= 1; c /= 2) {
            const bool fills = (int64_t)B * c >= num_sms;
            if ((int64_t)B * c <= capacity &&
                (c == 1 || ceil_div(V, c) >= (fills ? min_full : min_small))) {
                C = c;
                break;
            }
        }
    }
    out->cluster = C;
    out->group = 1;
    out->threads = nw * 32;
    out->smem_bytes = 0;
    out->slice = round_up(ceil_div(V, C), kSliceAlign);
    out->grid = (int64_t)B * C;
    out->bulk_copy = ((V * es) % 16) == 0 ? 1 : 0;
    out->prefetch_next = 0;
    out->stages = 0;  // no shared-memory ring
    return SV_OK;
}

}  // namespace

extern "C" int spec_verify_plan_greedy_for(int num_sms, int max_cluster, int B, int K, int64_t V,
                                           int logits_dtype, int ovr_cluster, sv_plan* out) {
    return plan_rows(num_sms, max_cluster, B, K, V, logits_dtype, ovr_cluster,
                     sv::kGreedyCtasPerSM, sv::kGreedyDepth, sv::kMaxCluster, out);
}

// Truncated-target verification: the same mapping with four resident CTAs
// per SM (its shared histograms), four loads in flight per lane, and
// clusters of at most eight CTAs.
extern "C" int spec_verify_plan_truncated_for(int num_sms, int max_cluster, int B, int K,
                                              int64_t V, int logits_dtype, int ovr_cluster,
                                              sv_plan* out) {
    return plan_rows(num_sms, max_cluster, B, K, V, logits_dtype, ovr_cluster,
                     sv::kTruncCtasPerSM, 4, sv::kTruncMaxCluster, out);
}

// Verification with draft logits: the truncated kernel's mapping when a
// filter is on; without filters the sampled verify's mapping (its kernel in
// the draft-logit form, 128 threads), with two rows of partials per group row
// and the per-CTA shared memory a GB300 CTA may opt into.
extern "C" int spec_verify_plan_draft_logits_for(int num_sms, int max_cluster, int B, int K,
                                                 int64_t V, int logits_dtype, int filters,
                                                 int ovr_cluster, sv_plan* out) {
    return filters ? plan_rows(num_sms, max_cluster, B, K, V, logits_dtype, ovr_cluster,
                               sv::kTruncCtasPerSM, 4, sv::kTruncMaxCluster, out)
                   : plan_impl(num_sms, sv::kSmemOptinPerCta, max_cluster, B, K, V, logits_dtype,
                               ovr_cluster, 0, 0, out, true);
}
