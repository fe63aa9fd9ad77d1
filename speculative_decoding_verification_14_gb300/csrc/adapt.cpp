// adapt.cpp -- acceptance telemetry read-out and the adaptive draft depth.
//
// The verify kernel can count, per call, how many sequences ended with each
// accepted length AL (1 .. K+1; bin 0 counts sequences that reported an
// error).  For one draft depth K those counts determine everything the pages
// ask to be watched:
//  * a sequence with AL <= K tested AL drafts and accepted AL - 1 of them;
//    one with AL = K + 1 tested and accepted all K;
//  * position i (0-based) was tested by every sequence with AL >= i + 1 and
//    accepted by every sequence with AL >= i + 2.
//
// [P1] reactapp.top, "Speculative decoding and early exit: speeding up
//      autoregressive decode", sections "Production perspective" (ship the
//      acceptance rate and the mean accepted length) and the operational
//      checklist (record acceptance histograms).
// [P2] trefon.com, "Decode is memory-bound: a ~59 tok/s ceiling on an RTX
//      4090 and how speculative decoding breaks it", section "Two things that
//      follow from the math" (cap the draft depth when the measured acceptance
//      falls below 35 %) and "Rules I follow" (pick the depth from measured
//      acceptance, keep measuring).
#include "../../include/spec_verify.h"

#include <cmath>
#include <cstring>

extern "C" int spec_adapt(const uint32_t* hist, int bins, int K, int K_max, int K_floor,
                          double threshold, uint64_t min_tested, sv_adapt* out) {
    if (!hist || !out || K < 0 || K > 32 || bins < K + 2 || K_max < 0 || K_max > 32 ||
        K_floor < 0 || K_floor > K_max || !(threshold >= 0.0 && threshold <= 1.0))
        return SV_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof *out);
    out->errors = hist[0];
    // reach[i] = sequences with AL >= i + 1 (i = 0 .. K)
    uint64_t reach[34] = {0};
    for (int n = K + 1; n >= 1; --n)
        reach[n - 1] = reach[n] + hist[n];
    out->sequences = reach[0];
    uint64_t al_sum = 0;
    for (int n = 1; n <= K + 1; ++n)
        al_sum += (uint64_t)n * hist[n];
    for (int i = 0; i < K; ++i) {
        out->tested += reach[i];
        out->accepted += reach[i + 1];
        out->pos_tested[i] = reach[i];
        out->pos_acceptance[i] = reach[i] ? (double)reach[i + 1] / (double)reach[i] : NAN;
    }
    for (int i = K; i < 32; ++i)
        out->pos_acceptance[i] = NAN;
    out->acceptance = out->tested ? (double)out->accepted / (double)out->tested : NAN;
    out->mean_accept_len = out->sequences ? (double)al_sum / (double)out->sequences : NAN;
    // The depth for the next passes: too few tests to judge keeps K; measured
    // acceptance below the threshold caps the depth at K_floor; otherwise the
    // full depth K_max.
    if (out->tested < min_tested || out->tested == 0)
        out->next_K = K < K_max ? K : K_max;
    else if (out->acceptance < threshold)
        out->next_K = K_floor;
    else
        out->next_K = K_max;
    return SV_OK;
}
