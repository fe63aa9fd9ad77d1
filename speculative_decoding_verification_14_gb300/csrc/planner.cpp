// planner.cpp -- maps one batched verify onto thread-block clusters.
//
// Work unit: one sequence b (its K+1 target rows, K draft rows, K tokens and
// K+1 uniforms) is verified by one cluster of C CTAs.  CTA r of the cluster
// owns the vocabulary slice [r*slice, (r+1)*slice) of every row of b, so the
// split-vocab partial softmax statistics of a row are combined inside the
// cluster through distributed shared memory; no global workspace and no
// second launch.
//
// Rows are loaded `group` at a time.  group = 1 reads only the rows the test
// loop reaches ([P1] "Speculative decoding: draft first, then verify": the
// loop stops at the first rejection), which minimises HBM bytes; it is chosen
// when the batch alone fills the GPU.  For small batches the pass is latency
// bound, so all K+1 rows are loaded at once (group = K+1) and decided from one
// cluster barrier.
//
// [P1] = reactapp.top, "Speculative decoding and early exit: speeding up
// autoregressive decode".
#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace {

int plan_impl(int num_sms, int smem_per_cta, int max_cluster, int B, int K, int64_t V, int dtype,
              int ovr_cluster, int ovr_group, int ovr_threads, sv_plan* out) {
    using namespace sv;
    if (!out || num_sms < 1 || smem_per_cta < 1 || max_cluster < 1 || B < 1 || K < 0 ||
        K > kMaxK || V < 1 || (dtype != SV_F32 && dtype != SV_BF16))
        return SV_ERR_INVALID_ARG;
    if (ovr_cluster < 0 || ovr_cluster > kMaxCluster || ovr_group < 0 ||
        (ovr_threads != 0 && ovr_threads != 128 && ovr_threads != 256 && ovr_threads != 512))
        return SV_ERR_INVALID_ARG;
    if (ovr_cluster > max_cluster)
        return SV_ERR_UNSUPPORTED;
    const int es = dtype == SV_BF16 ? 2 : 4;
    const int rows = K + 1;
    const int cmax = max_cluster < kMaxCluster ? max_cluster : kMaxCluster;
    const int threads = ovr_threads ? ovr_threads : 256;

    int C;
    if (ovr_cluster) {
        C = ovr_cluster;
    } else {
        // big clusters when the batch is small, so that a sequence's rows are
        // spread over many SMs; 8 (the portable size) otherwise
        C = (int64_t)B * 8 < 2 * (int64_t)num_sms ? 16 : 8;
        if (C > cmax)
            C = cmax;
        while (C > 1 && ceil_div(V, C) < kMinSlice)
            C /= 2;
    }
    int G;
    if (ovr_group)
        G = ovr_group < rows ? ovr_group : rows;
    else
        G = (int64_t)B * C >= 2 * (int64_t)num_sms ? 1 : rows;

    for (;;) {
        const int64_t slice = round_up(ceil_div(V, C), kSliceAlign);
        int64_t smem = smem_bytes_for(slice, es, G, threads);
        while (smem > smem_per_cta && G > 1 && !ovr_group) {
            G = (G + 1) / 2;
            smem = smem_bytes_for(slice, es, G, threads);
        }
        if (smem <= smem_per_cta) {
            out->cluster = C;
            out->group = G;
            out->threads = threads;
            out->smem_bytes = (int)smem;
            out->slice = slice;
            out->grid = (int64_t)B * C;
            out->bulk_copy = ((V * es) % 16) == 0 ? 1 : 0;
            out->prefetch_next = 0;
            return SV_OK;
        }
        if (ovr_cluster || C >= cmax)
            return SV_ERR_UNSUPPORTED;
        C *= 2;
        if (C > cmax)
            C = cmax;
    }
}

}  // namespace

extern "C" int spec_verify_plan_for(int num_sms, int smem_per_cta, int max_cluster, int B, int K,
                                    int64_t V, int logits_dtype, int ovr_cluster, int ovr_group,
                                    int ovr_threads, sv_plan* out) {
    return plan_impl(num_sms, smem_per_cta, max_cluster, B, K, V, logits_dtype, ovr_cluster,
                     ovr_group, ovr_threads, out);
}
