// truncated.cu -- verification against a truncated target distribution
// (top-p and min-p) for sm_103a.
//
// [P2] names the production sampler settings of its engine: temperature 0.6,
// top-p 0.95, min-p 0.05.  With such a sampler the target distribution of the
// verify step is p~ instead of p = softmax(l/T):
//   min-p keeps token v when p_v >= min_p * max p;
//   top-p keeps v when the mass of the tokens strictly more probable than v is
//         below top_p (every token tied at the boundary is kept);
//   p~ = p on the kept tokens, divided by their sum.
// Both filters look at the untruncated p, so their order does not matter.
// p~ then replaces p in every step of [P1]'s loop: the test u*q(x) < p~(x),
// the residual max(0, p~_j - q_j) and the bonus draw from p~_K.
//
// [P1] reactapp.top, "Speculative decoding and early exit: speeding up
//      autoregressive decode", section "Speculative decoding: draft first,
//      then verify".
// [P2] trefon.com, "Decode is memory-bound: a ~59 tok/s ceiling on an RTX
//      4090 and how speculative decoding breaks it", section "Two things that
//      follow from the math".
//
// Design: one cluster of C CTAs per sequence, vocabulary slices per CTA and
// stretches per warp, rows in order with the early stop.  Per row:
//  A. one pass for the row maximum l_max and S = sum 2^((l - l_max) c)
//     (c = log2(e)/T), pushed as warp partials to every CTA (st.async on an
//     mbarrier) and merged by every warp;
//  B. the top-p cut by radix selection over an order-preserving key of the
//     stored logits (two 8-bit levels for bf16, four for f32): each level is
//     one pass that bins the weights of the candidate tokens (min-p survivors
//     whose key matches the prefix chosen so far) into 256 shared-memory
//     bins, the CTA histograms are pushed to every CTA, and every warp finds
//     the digit where the mass above crosses top_p * S;
//  C. the test on x_i with p~(x_i) * E = 2^((l_x - l_max) c) for a kept x_i,
//     E the kept mass;
//  D. for the corrected or bonus token: a pass for per-warp weight totals,
//     pushed to every CTA; the warp that holds the crossing point walks its
//     stretch again to find the token and writes the outputs.
// Threshold decisions are taken on the stored logits: min-p as
// l - l_max >= T ln(min_p), top-p on the key, so the kept set depends on the
// weights only through the top-p masses.
//
// The same kernel verifies from the drafter's LOGITS d [B, K, V] instead of q
// (DL): [P1]'s loop forms q = softmax(d / T_d) itself.  Pass A then streams the
// target row and the draft row together and keeps both rows' statistics; the
// test uses q(x) S_d = 2^((d_x - d_max) c_d), and the draw's residual forms q
// from the draft row the same way.  (The untruncated draft-logit verify runs
// on the sampled verify's kernel instead.)
//
// Row passes load batches of 16-byte units per lane, sum them with packed
// arithmetic (one maximum test per batch), and ask L2 for the batch three
// ahead; the test's two values are asked into L2 when a row starts.
#include <cuda_runtime.h>
#include <cooperative_groups.h>

#include <cstdint>
#include <cstring>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kNT = 128;
constexpr int kNW = kNT / 32;
constexpr int kMaxC = sv::kTruncMaxCluster;
constexpr int kBins = 256;

struct TArgs {
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
    int B, K, C, vec;
    int qvec;        // 1: draft rows may be read as float4 (16-byte aligned rows)
    const void* dlogits;  // draft logits [B, K, V] (target dtype), or NULL: q given
    float c;         // log2(e) / T, rounded to float
    float cd;        // log2(e) / T_draft, rounded to float (draft logits)
    float T;
    float dmin;      // T * ln(min_p): min-p keeps l - l_max >= dmin (-inf: off)
    double top_p;    // >= 1: top-p off
    unsigned long long wait_ns;
};

// ------------------------------------------------------------------ PTX -----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect(unsigned long long* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Phase `parity` of `bar`, polled with a growing sleep; false after limit_ns.
__device__ __noinline__ bool mbar_wait_limited(unsigned long long* bar, uint32_t parity,
                                               unsigned long long limit_ns) {
    if (mbar_try(bar, parity))
        return true;
    const unsigned long long t0 = now_ns();
    unsigned sleep = 32;
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        __nanosleep(sleep);
        if (mbar_try(bar, parity))
            return true;
        if (sleep < 256)
            sleep <<= 1;
        if ((it & 15u) == 15u && now_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

// 16 bytes into the same slot of cluster CTA `rank`, counted on its `bar`.
__device__ __forceinline__ void push_v4(const void* slot, const void* bar, uint32_t rank, float4 v) {
    uint32_t d, m;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr(slot)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(m) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(d),
        "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
        "r"(__float_as_uint(v.w)), "r"(m)
        : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------- elements -----

// Entry e of a 16-byte vector of ES-byte logits, widened exactly to float.
template <int ES>
__device__ __forceinline__ float vec_entry(const uint4& v, int e) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (ES == 4) {
        return __uint_as_float(w[e]);
    } else {
        const uint32_t x = w[e >> 1];
        return __uint_as_float((e & 1) ? (x & 0xffff0000u) : (x << 16));
    }
}

// Order-preserving key of a stored logit (larger logit, larger key).
template <int ES>
__device__ __forceinline__ uint32_t key_of(float l) {
    uint32_t b = __float_as_uint(l);
    if constexpr (ES == 2)
        b >>= 16;
    constexpr uint32_t sign = ES == 2 ? 0x8000u : 0x80000000u;
    constexpr uint32_t all = ES == 2 ? 0xffffu : 0xffffffffu;
    return (b & sign) ? (b ^ all) : (b | sign);
}

__device__ __forceinline__ float load_entry(const void* base, int es, int64_t idx) {
    if (es == 4)
        return __ldg(static_cast<const float*>(base) + idx);
    const uint16_t h = __ldg(static_cast<const unsigned short*>(base) + idx);
    return __uint_as_float((uint32_t)h << 16);
}

// Kahan-style compensated accumulation (sum, compensation).
__device__ __forceinline__ void acc_add(float& s, float& comp, float x) {
    const float y = x - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

}  // namespace

namespace {

constexpr int kDepth = 4;     // 16-byte loads in flight per lane
constexpr int kChunks = 128;  // draw: chunk totals kept per warp

// Calls fn(l, e) for every entry of this warp's stretch of one row (e = entry
// index within the CTA's slice), lane by lane; entries of one lane come in
// increasing order, the lanes interleave by vector.
template <int ES>
__device__ __forceinline__ float vec_max(const uint4& w);  // below, with the packed helpers

// (vector path) unit_may(m) tells from a unit's largest entry m whether any
// of its entries can matter to fn; units it rules out are skipped whole.
template <int ES, typename U, typename F>
__device__ __forceinline__ void visit(const TArgs& a, int64_t row_elem, int64_t w0, int64_t w1,
                                      int lane, U&& unit_may, F&& fn) {
    constexpr int E = 16 / ES;
    if (a.vec) {
        const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.logits) +
                                                         row_elem * ES);
        for (int64_t base = w0; base < w1; base += 32 * kDepth) {
            uint4 r[kDepth];
#pragma unroll
            for (int k = 0; k < kDepth; ++k) {
                const int64_t idx = base + k * 32 + lane;
                if (idx < w1)
                    r[k] = ld_stream(rp + idx);
            }
#pragma unroll
            for (int k = 0; k < kDepth; ++k) {
                const int64_t idx = base + k * 32 + lane;
                if (idx < w1 && unit_may(vec_max<ES>(r[k]))) {
#pragma unroll
                    for (int t = 0; t < E; ++t)
                        fn(vec_entry<ES>(r[k], t), idx * E + t);
                }
            }
        }
    } else {
        for (int64_t e = w0 + lane; e < w1; e += 32)
            fn(load_entry(a.logits, ES, row_elem + e), e);
    }
}

__device__ __forceinline__ float fmax_nan(float x, float y) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(x), "f"(y));
    return d;
}

// ------------------------------------------------------ packed vectors -----
// A 16-byte vector of E = 16/ES logits taken with packed instructions: the
// NaN-propagating maximum (max.NaN.bf16x2 for bf16), l - m with a bf16
// operand widened exactly inside the subtraction (add.rn.f32.bf16), and f32x2
// multiplies and adds.  Entry 2h and 2h + 1 form pair h (the low and high
// halves of word h for bf16), the order vec_entry uses.

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// l - m for the two bf16 entries of a 32-bit word (nm = -m), each rounded once
__device__ __forceinline__ float2 bf16x2_minus(uint32_t w, float nm) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %3;\n\t"
        "add.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w), "f"(nm));
    return make_float2(lo, hi);
}

template <int ES>
__device__ __forceinline__ float vec_max(const uint4& w) {
    if constexpr (ES == 2) {
        const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w));
        return fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    } else {
        return fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                        fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

// d[h] = (entry 2h - m, entry 2h + 1 - m), nm = -m
template <int ES>
__device__ __forceinline__ void vec_minus(const uint4& w, float nm, float2 (&d)[8 / ES]) {
    if constexpr (ES == 2) {
        d[0] = bf16x2_minus(w.x, nm);
        d[1] = bf16x2_minus(w.y, nm);
        d[2] = bf16x2_minus(w.z, nm);
        d[3] = bf16x2_minus(w.w, nm);
    } else {
        const float2 n2 = make_float2(nm, nm);
        d[0] = __fadd2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), n2);
        d[1] = __fadd2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), n2);
    }
}

// A lane's running row statistics: its maximum mx and the compensated sum
// (sm, sc) of 2^((l - mx) c); bad once a NaN or +inf was seen.
struct LaneStats {
    float mx = -INFINITY, sm = 0.f, sc = 0.f;
    bool bad = false;
};

// One entry (element path): a rescale when it lies above the lane's maximum,
// then its term against the lane maximum.
__device__ __forceinline__ void lane_update_one(LaneStats& st, float l, float c) {
    if (l != l || l == INFINITY) {
        st.bad = true;
        return;
    }
    if (l == -INFINITY)  // weight 0
        return;
    if (l > st.mx) {
        const float f = ex2((st.mx - l) * c);
        st.sm *= f;
        st.sc *= f;
        st.mx = l;
    }
    acc_add(st.sm, st.sc, ex2((l - st.mx) * c));
}

// The warp's maximum and S = sum 2^((l - max) c) against it, from its lanes.
__device__ __forceinline__ void warp_finish(const LaneStats& st, float c, float& wmx, float& wsm,
                                            bool& wbad) {
    wmx = warp_max(st.mx);
    const float s = (st.mx > -INFINITY) ? (st.sm - st.sc) * ex2((st.mx - wmx) * c) : 0.f;
    wsm = warp_sum(s);
    wbad = __any_sync(kFull, st.bad);
}

// A batch of loaded units (ok[k]: unit k was loaded): the batch maximum, a
// rescale when it lies above the lane's maximum, then every term against the
// lane maximum with packed arithmetic and two packed accumulators.  Terms stay
// at most 1, as with one unit at a time, but the maximum is compared once per
// batch.  Returns the batch maximum.
template <int ES, int D>
__device__ __forceinline__ float lane_update_batch(LaneStats& st, const uint4 (&r)[D],
                                                  const bool (&ok)[D], float c) {
    float bm = -INFINITY;
#pragma unroll
    for (int k = 0; k < D; ++k)
        if (ok[k])
            bm = fmax_nan(bm, vec_max<ES>(r[k]));
    if (bm != bm || bm == INFINITY) {
        st.bad = true;
        return bm;
    }
    if (bm == -INFINITY)  // weights 0
        return bm;
    if (bm > st.mx) {
        const float f = ex2((st.mx - bm) * c);
        st.sm *= f;
        st.sc *= f;
        st.mx = bm;
    }
    const float2 c2 = make_float2(c, c);
    const float nm = -st.mx;
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < D; ++k) {
        if (ok[k]) {
            float2 d[8 / ES];
            vec_minus<ES>(r[k], nm, d);
#pragma unroll
            for (int h = 0; h < 8 / ES; ++h) {
                const float2 y = __fmul2_rn(d[h], c2);
                const float2 e = make_float2(ex2(y.x), ex2(y.y));
                if (h & 1)
                    s1 = __fadd2_rn(s1, e);
                else
                    s0 = __fadd2_rn(s0, e);
            }
        }
    }
    const float2 t = __fadd2_rn(s0, s1);
    acc_add(st.sm, st.sc, t.x + t.y);
    return bm;
}

// Loads of one batch: units b0 + k*32 + lane (k < D) of the stretch ending at
// w1; ok[k] tells which exist.
template <int D>
__device__ __forceinline__ void load_batch(const uint4* rp, int64_t b0, int64_t w1, int lane,
                                           uint4 (&r)[D], bool (&ok)[D]) {
    // 32-bit offsets inside the batch (a stretch holds far fewer than 2^31 units)
    const uint4* bp = rp + b0;
    const int64_t rem64 = w1 - b0;
    const int rem = rem64 < 32 * D ? (int)rem64 : 32 * D;
#pragma unroll
    for (int k = 0; k < D; ++k) {
        ok[k] = k * 32 + lane < rem;
        if (ok[k])
            r[k] = ld_stream(bp + (k * 32 + lane));
    }
}

// L2 lookahead for the batch loops: lane 0 asks L2 for the batch `kAhead`
// batches past b0 (one bulk prefetch of its contiguous units), so the loads
// of a batch find their lines in L2 instead of waiting a full DRAM latency.
// No registers are held for it, and nothing past the stretch is touched.
constexpr int kAhead = 3;

__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int D>
__device__ __forceinline__ void prefetch_batch(const uint4* rp, int64_t b, int64_t w1, int lane) {
    if (lane == 0 && b < w1) {
        const int64_t n = w1 - b < 32 * D ? w1 - b : 32 * D;
        prefetch_l2(rp + b, (uint32_t)(n * 16));
    }
}

// The prologue: batches 1 .. kAhead - 1 of the stretch.
template <int D>
__device__ __forceinline__ void prefetch_start(const uint4* rp, int64_t w0, int64_t w1, int lane) {
#pragma unroll
    for (int n = 1; n < kAhead; ++n)
        prefetch_batch<D>(rp, w0 + (int64_t)n * 32 * D, w1, lane);
}

// min-p survivor lists (truncated target with min-p on): per warp and row,
// and per CTA (the CTA's list travels with its count in one histogram slot).
constexpr int kCandW = 128;
constexpr int kCandC = 511;

// The largest entry of each group of batches of a warp's row pass, kept in
// shared memory (slots of `per` consecutive batches, at most kSlots of them),
// so that a later pass over the row can skip every group that cannot hold a
// min-p survivor.
constexpr int kSlots = 32;

struct SlotMax {
    float* slot;   // [kSlots], or null: not recorded
    int per;       // batches per slot
    int cnt = 0, s = 0;
    float run = -INFINITY;
    __device__ __forceinline__ void add(float lane_bm, bool last, int lane) {
        if (!slot)
            return;
        run = fmaxf(run, warp_max(lane_bm));
        if (++cnt == per || last) {
            if (lane == 0)
                slot[s] = run;
            ++s;
            cnt = 0;
            run = -INFINITY;
        }
    }
};

// One row's statistics over this warp's stretch of `base` (vector path; the
// element path takes one entry at a time), D loads in flight per lane.
template <int ES, int D>
__device__ __forceinline__ void warp_row_stats(const TArgs& a, const void* base, int64_t re,
                                               int64_t w0, int64_t w1, int lane, float c,
                                               float& wmx, float& wsm, bool& wbad,
                                               SlotMax* sm = nullptr) {
    LaneStats st;
    if (a.vec) {
        const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(base) +
                                                         re * ES);
        prefetch_start<D>(rp, w0, w1, lane);
        for (int64_t b0 = w0; b0 < w1; b0 += 32 * D) {
            prefetch_batch<D>(rp, b0 + kAhead * 32 * D, w1, lane);
            uint4 r[D];
            bool ok[D];
            load_batch<D>(rp, b0, w1, lane, r, ok);
            const float bm = lane_update_batch<ES, D>(st, r, ok, c);
            if (sm)
                sm->add(bm, b0 + 32 * D >= w1, lane);
        }
    } else {
        for (int64_t e = w0 + lane; e < w1; e += 32) {
            lane_update_one(st, load_entry(base, ES, re + e), c);
        }
    }
    warp_finish(st, c, wmx, wsm, wbad);
}

// The target row and the draft row together (vector path): both rows' units
// come in one loop, D deep each, so a lane has 2 D loads in flight.
template <int ES, int D>
__device__ __forceinline__ void warp_row_stats_pair(const void* tbase, int64_t tre,
                                                    const void* dbase, int64_t dre, int64_t w0,
                                                    int64_t w1, int lane, float c, float cd,
                                                    float& wmx, float& wsm, bool& wbad,
                                                    float& dmx, float& dsm, bool& dbad,
                                                    SlotMax* sm = nullptr) {
    const uint4* tp = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(tbase) +
                                                     tre * ES);
    const uint4* dp = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(dbase) +
                                                     dre * ES);
    LaneStats st, sd;
    prefetch_start<D>(tp, w0, w1, lane);
    prefetch_start<D>(dp, w0, w1, lane);
    for (int64_t b0 = w0; b0 < w1; b0 += 32 * D) {
        prefetch_batch<D>(tp, b0 + kAhead * 32 * D, w1, lane);
        prefetch_batch<D>(dp, b0 + kAhead * 32 * D, w1, lane);
        uint4 rt[D], rd[D];
        bool ok[D];
        load_batch<D>(tp, b0, w1, lane, rt, ok);
        load_batch<D>(dp, b0, w1, lane, rd, ok);
        const float bm = lane_update_batch<ES, D>(st, rt, ok, c);
        lane_update_batch<ES, D>(sd, rd, ok, cd);
        if (sm)
            sm->add(bm, b0 + 32 * D >= w1, lane);
    }
    warp_finish(st, c, wmx, wsm, wbad);
    warp_finish(sd, cd, dmx, dsm, dbad);
}

// DL: draft logits instead of draft probabilities (q_i = softmax(d_i / T_d),
// formed here from the draft row's own statistics).
template <int ES, bool DL>
__global__ void __launch_bounds__(kNT, sv::kTruncCtasPerSM)
    sv_trunc_kernel(const __grid_constant__ TArgs a) {
    constexpr int E = 16 / ES;
    constexpr int KEYBITS = 8 * ES;
    constexpr int LEVELS = KEYBITS / 8;
    constexpr int MC = kMaxC;  // largest cluster
    constexpr int HB = kBins;  // histogram bins held
    constexpr int HC = kMaxC;
    // row pass: loads in flight per lane and row (a target row alone, or the
    // target and draft rows together: deeper pairs spill registers)
    constexpr int DA = DL ? kDepth : 8;
    constexpr int DP = 4;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)a.C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, C = a.C;
    const int P = C * kNW;
    const int64_t V = a.V;
    const float c = a.c;
    const bool use_min = a.dmin > -INFINITY;
    const bool use_top = a.top_p < 1.0;
    // min-p bounds the kept set: one pass lists the survivors of a row and
    // the top-p cut is taken over those lists (aligned rows)
    const bool list_ok = use_min && a.vec;

    __shared__ __align__(16) float4 part[2][MC * kNW];          // warp partials, by use parity
    // top-p histograms hold fixed-point masses: weights 2^((l - l_max) c) <= 1
    // scaled by 2^fix and rounded to integers, so the adds are exact and their
    // order does not matter
    __shared__ __align__(16) unsigned long long hrecv[2][HC][HB];  // CTA histograms, by use parity
    __shared__ __align__(16) unsigned long long hloc[HB];          // this CTA's histogram
    __shared__ __align__(8) unsigned long long xbar[2], hbar[2];
    __shared__ int xs[sv::kMaxK];
    __shared__ float us[sv::kMaxRows];
    __shared__ float rsm[sv::kMaxRows], rss[sv::kMaxRows], pdr[sv::kMaxK];
    __shared__ float ctot[kNW][kChunks];                         // draw: chunk totals per warp
    // min-p survivors: each warp's, then the CTA's (values and entry
    // indices); the draw over a listed row reuses them
    constexpr int CW = kCandW, CC = kCandC;
    __shared__ float cw_v[kNW][CW];
    __shared__ int cw_i[kNW][CW];
    __shared__ int cw_n[kNW];
    __shared__ float cl_v[CC];
    __shared__ int cl_i[CC];
    __shared__ int cl_cnt[kNW];
    __shared__ float smax[kNW][kSlots];                         // row pass: group maxima

    const int64_t v0 = (int64_t)rank * a.slice;
    const int64_t L = v0 < V ? (V - v0 < a.slice ? V - v0 : a.slice) : 0;
    const int64_t row0 = (int64_t)b * (K + 1);
    const int64_t units = a.vec ? L / E : L;
    const int64_t per_w = (units + kNW - 1) / kNW;
    const int64_t w0 = per_w * warp < units ? per_w * warp : units;
    const int64_t w1 = w0 + per_w < units ? w0 + per_w : units;

    if (tid == 0) {
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        mbar_init(&hbar[0], 1);
        mbar_init(&hbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < K)
        xs[tid] = a.tokens[(int64_t)b * K + tid];
    if (tid <= K)
        us[tid] = a.u[row0 + tid];
    if (tid < kNW)
        cw_n[tid] = 0;
    __syncthreads();
    cluster_arrive();
    bool ready = false;
    int state = SV_OK;
    {
        const bool bad_x = __any_sync(kFull, lane < K && (xs[lane] < 0 || (int64_t)xs[lane] >= V));
        const float ul = lane <= K ? us[lane] : 0.5f;
        const float uh = (lane == 0 && K == sv::kMaxK) ? us[sv::kMaxK] : 0.5f;
        const bool bad_u = __any_sync(kFull, !(ul >= 0.f && ul < 1.f) || !(uh >= 0.f && uh < 1.f));
        if (bad_x)
            state = SV_ERR_TOKEN_RANGE;
        else if (bad_u)
            state = SV_ERR_UNIFORM_RANGE;
    }

    uint32_t xcnt = 0, hcnt = 0;  // exchanges so far (slot = cnt & 1, phase = (cnt >> 1) & 1)
    // Every warp pushes one float4 to slot (rank, warp) of every CTA and gets
    // back all P of them in part[slot]; false if they did not come in time.
    auto exchange = [&](float4 v) -> int {
        const int s = (int)(xcnt & 1u);
        const uint32_t ph = (xcnt >> 1) & 1u;
        ++xcnt;
        if (!ready) {
            cluster_wait();
            ready = true;
        }
        if (tid == 0)
            mbar_expect(&xbar[s], (uint32_t)(P * 16));
        if (lane < C)
            push_v4(&part[s][rank * kNW + warp], &xbar[s], (uint32_t)lane, v);
        // (every thread of the CTA takes the same outcome, so control flow
        // stays uniform even when a wait runs out)
        const int ok = __syncthreads_and(mbar_wait_limited(&xbar[s], ph, a.wait_ns) ? 1 : 0);
        return ok ? s : -1;
    };
    // The CTA histogram hloc goes to slot (rank) of every CTA; every warp then
    // sees all C of them in hrecv[slot].
    auto exchange_hist = [&]() -> int {
        const int s = (int)(hcnt & 1u);
        const uint32_t ph = (hcnt >> 1) & 1u;
        ++hcnt;
        if (!ready) {
            cluster_wait();
            ready = true;
        }
        __syncthreads();  // hloc complete
        if (tid == 0)
            mbar_expect(&hbar[s], (uint32_t)(C * kBins * 8));
        for (int idx = tid; idx < C * (kBins / 2); idx += kNT) {
            const int d = idx / (kBins / 2), k = idx % (kBins / 2);
            push_v4(&hrecv[s][rank][k * 2], &hbar[s], (uint32_t)d,
                    reinterpret_cast<const float4*>(hloc)[k]);
        }
        // (one outcome for the whole CTA; also: hloc is read by everyone
        // before it is cleared again)
        const int ok = __syncthreads_and(mbar_wait_limited(&hbar[s], ph, a.wait_ns) ? 1 : 0);
        return ok ? s : -1;
    };

    int j = -1;
    bool listed = false;                  // the decided row's kept set came from its survivor list
    int ncl = 0;                          // ... this CTA's survivors in cl_v / cl_i
    float lmax = 0.f, E_kept = 0.f;       // the decided row's statistics
    float dmax = 0.f, dS = 0.f;           // ... and its draft row's (draft logits)
    uint32_t key_t = 0;                   // top-p: kept keys are >= key_t
    for (int i = 0; i <= K && state == SV_OK; ++i) {
        const int64_t re = (row0 + i) * V + v0;  // first element of this CTA's slice of row i
        // the test's two values (l_x and the draft's d_x or q(x)) sit at random
        // positions: ask L2 for them now, so the test after the exchange does
        // not wait a DRAM latency
        if (i < K && lane == 0) {
            const int64_t xi = (int64_t)xs[i];
            prefetch_line_l2(static_cast<const unsigned char*>(a.logits) + ((row0 + i) * V + xi) * ES);
            if constexpr (DL)
                prefetch_line_l2(static_cast<const unsigned char*>(a.dlogits) +
                                 (((int64_t)b * K + i) * V + xi) * ES);
            else
                prefetch_line_l2(a.q + ((int64_t)b * K + i) * V + xi);
        }
        // ---- A: row maximum and S = sum 2^((l - l_max) c); with draft
        // logits, the same for the draft row d_i at c_d (i < K) ----
        // (partial: (max, S or -1 when bad, draft max, draft S or -1))
        float wmx, wsm, dmx = -INFINITY, dsm = 0.f;
        bool bad, dbad = false;
        // (with min-p lists: the largest entry of every slot of batches)
        const int batch_u = 32 * ((DL && i < K && a.vec) ? DP : DA);
        const int nbat = (int)((w1 - w0 + batch_u - 1) / batch_u);
        const int per = (nbat + kSlots - 1) / kSlots > 0 ? (nbat + kSlots - 1) / kSlots : 1;
        SlotMax slm{list_ok ? smax[warp] : nullptr, per};
        if (DL && i < K && a.vec) {
            warp_row_stats_pair<ES, DP>(a.logits, re, a.dlogits, ((int64_t)b * K + i) * V + v0, w0,
                                        w1, lane, c, a.cd, wmx, wsm, bad, dmx, dsm, dbad, &slm);
        } else {
            warp_row_stats<ES, DA>(a, a.logits, re, w0, w1, lane, c, wmx, wsm, bad, &slm);
            if (DL && i < K)
                warp_row_stats<ES, DA>(a, a.dlogits, ((int64_t)b * K + i) * V + v0, w0, w1, lane,
                                       a.cd, dmx, dsm, dbad);
        }
        const int s1 = exchange(make_float4(wmx, bad ? -1.f : wsm, dmx, dbad ? -1.f : dsm));
        if (s1 < 0) {
            state = SV_ERR_TIMEOUT;
            break;
        }
        {
            // merged in a fixed order, so every warp holds the same statistics
            float m = -INFINITY, md = -INFINITY;
            bool bd = false;
            for (int p = lane; p < P; p += 32) {
                const float4 q4 = part[s1][p];
                m = fmaxf(m, q4.x);
                md = fmaxf(md, q4.z);
                bd = bd || q4.y < 0.f || q4.w < 0.f;
            }
            m = warp_max(m);
            md = warp_max(md);
            // each lane rescales its partials, one butterfly sums them (the
            // same order in every warp)
            float S = 0.f, Sd = 0.f;
            for (int p = lane; p < P; p += 32) {
                const float4 q4 = part[s1][p];
                if (q4.x > -INFINITY)
                    S += q4.y * ex2((q4.x - m) * c);
                if (DL && q4.z > -INFINITY)
                    Sd += q4.w * ex2((q4.z - md) * a.cd);
            }
            S = warp_sum(S);
            if constexpr (DL)
                Sd = warp_sum(Sd);
            if (__any_sync(kFull, bd) || !(m > -INFINITY) || (DL && i < K && !(md > -INFINITY))) {
                state = SV_ERR_NONFINITE;
                break;
            }
            lmax = m;
            E_kept = S;
            dmax = md;
            dS = Sd;
            if (lane == 0 && warp == 0) {
                rsm[i] = __fdiv_rn(m, a.T);
                rss[i] = S;
            }
        }
        const float S_all = E_kept;
        key_t = 0;
        listed = false;
        // ---- B: the kept set ----
        if (use_min || use_top) {
            // fixed point: 2^fix per unit weight, with fix chosen so that V
            // weights of at most 1 sum below 2^63 (44 bits for V <= 2^18);
            // each weight is off by at most 2^-(fix+1) after rounding
            const int vbits = 64 - __clzll((unsigned long long)(V > 1 ? V - 1 : 1));
            const int fix = min(44, 62 - vbits);
            const float fscale = __int_as_float((127 + fix) << 23);      // 2^fix
            const float funscale = __int_as_float((127 - fix) << 23);    // 2^-fix
            const unsigned long long thr =
                (unsigned long long)(a.top_p * (double)S_all * (double)fscale);
            // With min-p on, one pass over the row lists its survivors
            // (l - l_max >= T ln(min_p)); they are compacted per CTA (warp
            // order, then the order found) and exchanged as values, and the cut
            // is taken over the union of the lists in every CTA alike, with the
            // same histograms as over the whole row.  A list past its capacity
            // anywhere sends every CTA through the histogram passes instead.
            int sL = -1;
            if (list_ok) {
                // only the slots of batches whose largest entry passes min-p
                const int64_t su = (int64_t)slm.per * batch_u;  // units per slot
                for (int sl = 0; sl < slm.s; ++sl) {
                    if (!(smax[warp][sl] - lmax >= a.dmin))
                        continue;
                    const int64_t u0 = w0 + sl * su;
                    visit<ES>(a, re, u0, u0 + su < w1 ? u0 + su : w1, lane,
                              [&](float um) -> bool { return um - lmax >= a.dmin; },
                              [&](float l, int64_t e) {
                                  if (l - lmax >= a.dmin) {
                                      const int pos = atomicAdd(&cw_n[warp], 1);
                                      if (pos < kCandW) {
                                          cw_v[warp][pos] = l;
                                          cw_i[warp][pos] = (int)e;
                                      }
                                  }
                              });
                }
                __syncwarp();
                const int nw = cw_n[warp];
                if (lane == 0)
                    cl_cnt[warp] = nw <= kCandW ? nw : -1;
                __syncthreads();
                int off = 0, tot = 0;
                bool ovf = false;
                for (int w2 = 0; w2 < kNW; ++w2) {
                    const int c2 = cl_cnt[w2];
                    ovf = ovf || c2 < 0;
                    off += (w2 < warp && c2 > 0) ? c2 : 0;
                    tot += c2 > 0 ? c2 : 0;
                }
                ovf = ovf || tot > kCandC;
                if (!ovf)
                    for (int k = lane; k < nw; k += 32) {
                        cl_v[off + k] = cw_v[warp][k];
                        cl_i[off + k] = cw_i[warp][k];
                    }
                if (lane == 0)
                    cw_n[warp] = 0;  // the next row lists afresh
                ncl = ovf ? 0 : tot;
                __syncthreads();     // the CTA's list is complete
                float* stg = reinterpret_cast<float*>(hloc);  // [count or -1, values]
                for (int k = tid; k <= ncl; k += kNT)
                    stg[k] = k == 0 ? (ovf ? -1.f : (float)tot) : cl_v[k - 1];
                sL = exchange_hist();
                if (sL < 0) {
                    state = SV_ERR_TIMEOUT;
                    break;
                }
                bool any_ovf = false;
                int nall = 0;
                for (int r = 0; r < C; ++r) {
                    const float cr = reinterpret_cast<const float*>(hrecv[sL][r])[0];
                    any_ovf = any_ovf || cr < 0.f;
                    nall += cr > 0.f ? (int)cr : 0;
                }
                listed = !any_ovf;
                if (listed && nall <= 64) {
                    // A short union: every warp takes the cut itself.  Lane l
                    // holds survivors l and l + 32 (in CTA order); a survivor is
                    // kept when the fixed-point mass of the survivors with a
                    // larger key is below top_p * S -- the same integers, and
                    // so the same kept set and E, as the histogram levels give.
                    float vv[2];
                    uint32_t kk[2];
                    unsigned long long ww[2], ab[2] = {0ull, 0ull};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int f = lane + 32 * h;
                        vv[h] = -INFINITY;
                        for (int r = 0, base = 0; r < C; ++r) {
                            const float* lv = reinterpret_cast<const float*>(hrecv[sL][r]);
                            const int nr = (int)lv[0];
                            if (f >= base && f < base + nr)
                                vv[h] = lv[1 + f - base];
                            base += nr;
                        }
                        kk[h] = f < nall ? key_of<ES>(vv[h]) : 0u;
                        ww[h] = f < nall ? __float2ull_rn(ex2((vv[h] - lmax) * c) * fscale) : 0ull;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        for (int src = 0; src < 32; ++src) {
                            const uint32_t ks = __shfl_sync(kFull, kk[h], src);
                            const unsigned long long ws = __shfl_sync(kFull, ww[h], src);
                            ab[0] += ks > kk[0] ? ws : 0ull;
                            ab[1] += ks > kk[1] ? ws : 0ull;
                        }
                    unsigned long long ek = 0;
                    uint32_t kmin = 0xffffffffu;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (lane + 32 * h < nall && (!use_top || ab[h] < thr)) {
                            ek += ww[h];
                            kmin = min(kmin, kk[h]);
                        }
#pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        ek += __shfl_xor_sync(kFull, ek, o);
                        kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
                    }
                    E_kept = __ull2float_rn(ek) * funscale;
                    key_t = use_top && nall > 0 ? kmin : 0u;
                    if (lane == 0)
                        cw_n[warp] = 0;  // (already clear; keeps the lists' state uniform)
                    goto cut_done;
                }
            }
            {
            uint32_t prefix = 0;
            unsigned long long above = 0;  // mass of candidates with keys above the prefix group
            for (int lev = 0; lev < LEVELS; ++lev) {
                for (int k = tid; k < kBins; k += kNT)
                    hloc[k] = 0ull;
                __syncthreads();
                const int sh_hi = KEYBITS - 8 * lev;   // prefix = key >> sh_hi
                const int sh_lo = KEYBITS - 8 * (lev + 1);
                // a unit can hold a candidate only if its largest entry passes
                // min-p and, past the first level, its key prefix is not below
                // the chosen one (keys order like the logits)
                const auto unit_may = [&](float um) -> bool {
                    if (use_min && !(um - lmax >= a.dmin))
                        return false;
                    return lev == 0 || (key_of<ES>(um) >> sh_hi) >= prefix;
                };
                int s2 = -1;
                if (listed) {
                    // the union of the survivor lists, every CTA the same
                    for (int r = 0; r < C; ++r) {
                        const float* lv = reinterpret_cast<const float*>(hrecv[sL][r]);
                        const int nr = (int)lv[0];
                        for (int k = tid; k < nr; k += kNT) {
                            const float l = lv[1 + k];
                            const uint32_t key = key_of<ES>(l);
                            if (lev > 0 && (key >> sh_hi) != prefix)
                                continue;
                            atomicAdd(&hloc[(key >> sh_lo) & 0xffu],
                                      __float2ull_rn(ex2((l - lmax) * c) * fscale));
                        }
                    }
                    __syncthreads();
                } else {
                    visit<ES>(a, re, w0, w1, lane, unit_may, [&](float l, int64_t) {
                        if (use_min && !(l - lmax >= a.dmin))
                            return;
                        const uint32_t key = key_of<ES>(l);
                        if (lev > 0 && (key >> sh_hi) != prefix)
                            return;
                        atomicAdd(&hloc[(key >> sh_lo) & 0xffu],
                                  __float2ull_rn(ex2((l - lmax) * c) * fscale));
                    });
                    s2 = exchange_hist();
                    if (s2 < 0) {
                        state = SV_ERR_TIMEOUT;
                        break;
                    }
                }
                // lane l holds bins 8l .. 8l+7, summed over the CTAs in a fixed order
                unsigned long long bin[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    unsigned long long acc = 0;
                    if (listed)
                        acc = hloc[lane * 8 + t];
                    else
                        for (int r = 0; r < C; ++r)
                            acc += hrecv[s2][r][lane * 8 + t];
                    bin[t] = acc;
                }
                unsigned long long lt = 0;
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    lt += bin[t];
                // mass of the bins of this and higher lanes (suffix sum over lanes)
                unsigned long long incl = lt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long v = __shfl_down_sync(kFull, incl, o);
                    if (lane + o < 32)
                        incl += v;
                }
                const unsigned long long above_lane = incl - lt;
                const unsigned long long total = __shfl_sync(kFull, incl, 0);
                if (lev == 0 && (!use_top || total < thr)) {
                    // min-p alone, or candidates holding less than top_p: all kept
                    E_kept = __ull2float_rn(total) * funscale;
                    break;
                }
                // the lowest non-empty digit whose mass above is below thr
                int hc = -1;
                unsigned long long hab = 0, hb = 0;
                unsigned long long run = above + above_lane;
#pragma unroll
                for (int t = 7; t >= 0; --t) {
                    if (bin[t] > 0 && run < thr) {
                        hc = lane * 8 + t;
                        hab = run;
                        hb = bin[t];
                    }
                    run += bin[t];
                }
                int best = hc < 0 ? 0x7fffffff : hc;
#pragma unroll
                for (int o = 16; o; o >>= 1)
                    best = min(best, __shfl_xor_sync(kFull, best, o));
                if (best == 0x7fffffff) {  // no digit below the cut: cannot happen for S > 0
                    state = SV_ERR_NONFINITE;
                    break;
                }
                const int src = best >> 3;
                hab = __shfl_sync(kFull, hab, src);
                hb = __shfl_sync(kFull, hb, src);
                prefix = (prefix << 8) | (uint32_t)best;
                above = hab;
                E_kept = __ull2float_rn(hab + hb) * funscale;
                if (lev == LEVELS - 1)
                    key_t = prefix;
                if (listed)
                    __syncthreads();  // every warp has read the bins before they are cleared
            }
            if (state != SV_OK)
                break;
            if (!use_top)
                key_t = 0;
            }
        cut_done:;
        }
        // ---- C: the test at position i ([P1]) ----
        if (i < K) {
            const int x = xs[i];
            const float lx = load_entry(a.logits, ES, (row0 + i) * V + x);
            const bool kept = (!use_min || lx - lmax >= a.dmin) && key_of<ES>(lx) >= key_t;
            if constexpr (DL) {
                // p~(x) E = 2^((l_x - l_max) c) and q(x) S_d = 2^((d_x - d_max) c_d), so
                // u q(x) < p~(x) <=> u E < 2^y S_d with y = (l_x - l_max) c - (d_x - d_max) c_d.
                // y is exact in double (products of two floats); 2^y = 2^n 2^f with one
                // float exp2 of the fraction, so the test has one rounded exponential
                // and no double transcendental.  Lane 0 decides, the warp follows.
                const float dx = load_entry(a.dlogits, ES, ((int64_t)b * K + i) * V + x);
                int acc = 0;
                if (lane == 0) {
                    if (!kept || lx == -INFINITY) {
                        acc = 0;  // p~(x) = 0
                    } else if (dx == -INFINITY) {
                        acc = 1;  // q(x) = 0 < p~(x)
                    } else {
                        double y = (double)(lx - lmax) * (double)c - (double)(dx - dmax) * (double)a.cd;
                        y = fmin(fmax(y, -4000.0), 4000.0);  // beyond: 2^y is 0 or inf in double
                        const double n = floor(y);
                        const float m = exp2f((float)(y - n));
                        acc = (double)us[i] * (double)E_kept < ldexp((double)m * (double)dS, (int)n);
                    }
                    if (warp == 0)
                        pdr[i] = kept ? __fdiv_rn(ex2((lx - lmax) * c), E_kept) : 0.f;
                }
                if (__shfl_sync(kFull, acc, 0))
                    continue;  // accepted
            } else {
                const float ex = kept ? ex2((lx - lmax) * c) : 0.f;
                const float qx = __ldg(a.q + ((int64_t)b * K + i) * V + x);
                if (!(qx >= 0.f && qx < INFINITY)) {
                    state = SV_ERR_NONFINITE;
                    break;
                }
                if (lane == 0 && warp == 0)
                    pdr[i] = __fdiv_rn(ex, E_kept);
                if (us[i] * qx * E_kept < ex)
                    continue;  // accepted
            }
        }
        j = i;
        break;
    }

    // ---- D: the corrected (j < K) or bonus (j = K) token, from p~ ([P1]) ----
    if (state == SV_OK) {
        const bool resid = j < K;
        const int64_t re = (row0 + j) * V + v0;
        const float* qrow = (resid && !DL) ? a.q + ((int64_t)b * K + j) * V + v0 : nullptr;
        const int64_t dre = ((int64_t)b * K + j) * V + v0;  // draft logits: row j's slice
        const uint4* dp = DL && resid ? reinterpret_cast<const uint4*>(
                                            static_cast<const unsigned char*>(a.dlogits) + dre * ES)
                                      : nullptr;
        // draft logits: q_v E = 2^((d_v - d_max) c_d) * (E / S_d)
        const float rq = DL && resid ? __fdiv_rn(E_kept, dS) : 0.f;
        const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.logits) +
                                                         re * ES);
        const float Ek = E_kept;
        bool fallback = false;
        // whether a token is kept, and 2^((l - l_max) c) for a kept token, 0
        // for a dropped one
        auto is_kept = [&](float l) -> bool {
            return l > -INFINITY && (!use_min || l - lmax >= a.dmin) && key_of<ES>(l) >= key_t;
        };
        auto kept_w = [&](float l) -> float { return is_kept(l) ? ex2((l - lmax) * c) : 0.f; };
        // with a filter on, q_j is read only at kept tokens (the residual is
        // zero elsewhere) and checked there alone
        const bool filt = use_min || use_top;
        // The stretch is walked in steps of 32 units (one per lane); g steps
        // make a chunk, whose total is kept in shared memory for the locate.
        const int64_t nsub = (w1 - w0 + 31) / 32;
        const int64_t g = nsub > 0 ? (nsub + kChunks - 1) / kChunks : 1;
        const int nch = (int)((nsub + g - 1) / g);
        const int U = a.vec ? E : 1;  // entries per unit
        // the lane's unit of step st: logits and (residual) draft probabilities
        auto load_unit = [&](int64_t st, float (&l)[E], float (&qv)[E]) -> bool {
            const int64_t ui = w0 + st * 32 + lane;
            if (ui >= w1)
                return false;
            if (a.vec) {
                const uint4 r = ld_stream(rp + ui);
#pragma unroll
                for (int t = 0; t < E; ++t)
                    l[t] = vec_entry<ES>(r, t);
            } else {
                l[0] = load_entry(a.logits, ES, re + ui);
            }
            if (DL && resid && !fallback) {
                if (a.vec) {
                    const uint4 r = ld_stream(dp + ui);
#pragma unroll
                    for (int t = 0; t < E; ++t)
                        qv[t] = vec_entry<ES>(r, t);
                } else {
                    qv[0] = load_entry(a.dlogits, ES, dre + ui);
                }
            } else if (resid && !fallback) {
                if (a.vec && a.qvec) {
                    const float4* q4 = reinterpret_cast<const float4*>(qrow + ui * E);
#pragma unroll
                    for (int h = 0; h < E / 4; ++h) {
                        const float4 v4 = __ldg(q4 + h);
                        qv[4 * h] = v4.x;
                        qv[4 * h + 1] = v4.y;
                        qv[4 * h + 2] = v4.z;
                        qv[4 * h + 3] = v4.w;
                    }
                } else {
                    for (int t = 0; t < U; ++t)
                        qv[t] = __ldg(qrow + ui * U + t);
                }
            }
            return true;
        };
        // weights (scaled by E): max(0, e - q E) for the residual, e for the
        // bonus row or the fallback to p~_j; returns their sum
        auto unit_weights = [&](const float (&l)[E], const float (&qv)[E], float (&w)[E],
                                bool& badq) -> float {
            float sum = 0.f;
            for (int t = 0; t < U; ++t) {
                const float ev = kept_w(l[t]);
                if (DL && resid && !fallback) {
                    // qv holds the draft logits (checked when the row was read)
                    w[t] = fmaxf(ev - ex2((qv[t] - dmax) * a.cd) * rq, 0.f);
                } else if (resid && !fallback) {
                    if (!(qv[t] >= 0.f && qv[t] < INFINITY) && (!filt || is_kept(l[t])))
                        badq = true;
                    w[t] = fmaxf(ev - qv[t] * Ek, 0.f);
                } else {
                    w[t] = ev;
                }
                sum += w[t];
            }
            return sum;
        };
        float cum_before = 0.f, Sw = 0.f, t = 0.f;
        int owner = -1;
        // draft logits, vector path: the draw's row pair (or the target row
        // alone for the bonus row and the fallback) stays in registers, DD
        // units deep; the weights are the bits unit_weights gives (the locate
        // re-derives them that way).
        const auto unit_weights_raw = [&](const uint4& lr, const uint4& dr, bool two) -> float {
            float sum = 0.f;
#pragma unroll
            for (int t = 0; t < E; ++t) {
                const float ev = kept_w(vec_entry<ES>(lr, t));
                sum += two ? fmaxf(ev - ex2((vec_entry<ES>(dr, t) - dmax) * a.cd) * rq, 0.f) : ev;
            }
            return sum;
        };
        const int g32 = (int)g;  // steps per chunk (chunk ends counted, not divided)
        // A listed row: p~_j is zero outside the survivors with keys >= key_t,
        // so max(0, p~_j - q_j) and p~_j are too, and the draw's weights are
        // those of the survivors alone, sorted into vocabulary order here
        // (into cw_v / cw_i); q or the draft logit is read, and q checked, at
        // the kept entries only.
        float* sv_v = &cw_v[0][0];
        int* sv_i = &cw_i[0][0];
        if (listed) {
            for (int k = tid; k < ncl; k += kNT) {
                const int ik = cl_i[k];
                int r = 0;
                for (int m = 0; m < ncl; ++m)
                    r += cl_i[m] < ik ? 1 : 0;
                sv_v[r] = cl_v[k];
                sv_i[r] = ik;
            }
            __syncthreads();
        }
        for (int round = 0; round < 2; ++round) {
            float wt = 0.f, wtc = 0.f, cpart = 0.f;
            bool badq = false;
            int gcnt = 0, chunk = 0;
            if (listed) {
                if (warp == 0) {
                    // weights (scaled by E) in vocabulary order, kept in cl_v
                    for (int k0 = 0; k0 < ncl; k0 += 32) {
                        const int k = k0 + lane;
                        float w = 0.f;
                        if (k < ncl) {
                            const float l = sv_v[k];
                            const bool kept = key_of<ES>(l) >= key_t;
                            const float ev = kept ? ex2((l - lmax) * c) : 0.f;
                            if (DL && resid && !fallback) {
                                w = fmaxf(ev - ex2((load_entry(a.dlogits, ES, dre + sv_i[k]) - dmax) *
                                                   a.cd) * rq, 0.f);
                            } else if (resid && !fallback && kept) {
                                const float qv = __ldg(qrow + sv_i[k]);
                                badq = badq || !(qv >= 0.f && qv < INFINITY);
                                w = fmaxf(ev - qv * Ek, 0.f);
                            } else if (!resid || fallback) {
                                w = ev;
                            }
                            cl_v[k] = w;
                        }
                        acc_add(wt, wtc, warp_sum(w));
                    }
                }
            }
            if constexpr (DL) if (a.vec && !listed) {
                constexpr int DD = 8;
                const bool two = resid && !fallback;
                // the steps st0 .. st0 + DD - 1 are units w0 + st * 32 + lane: one
                // contiguous batch of DD * 32 units, as in the row loops
                prefetch_start<DD>(rp, w0, w1, lane);
                if (two)
                    prefetch_start<DD>(dp, w0, w1, lane);
                for (int64_t st0 = 0; st0 < nsub; st0 += DD) {
                    prefetch_batch<DD>(rp, w0 + (st0 + kAhead * DD) * 32, w1, lane);
                    if (two)
                        prefetch_batch<DD>(dp, w0 + (st0 + kAhead * DD) * 32, w1, lane);
                    uint4 lr[DD], dr[DD];
#pragma unroll
                    for (int k = 0; k < DD; ++k) {
                        const int64_t ui = w0 + (st0 + k) * 32 + lane;
                        if (st0 + k < nsub && ui < w1) {
                            lr[k] = ld_stream(rp + ui);
                            if (two)
                                dr[k] = ld_stream(dp + ui);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < DD; ++k) {
                        const int64_t st = st0 + k;
                        if (st >= nsub)
                            break;
                        if (w0 + st * 32 + lane < w1) {
                            cpart += unit_weights_raw(lr[k], dr[k], two);
                        }
                        if (++gcnt == g32 || st + 1 == nsub) {  // chunk `chunk` ends here
                            const float ct = warp_sum(cpart);
                            cpart = 0.f;
                            if (lane == 0)
                                ctot[warp][chunk] = ct;
                            ++chunk;
                            gcnt = 0;
                            acc_add(wt, wtc, ct);
                        }
                    }
                }
            }
            for (int64_t st0 = 0; st0 < (((DL && a.vec) || listed) ? 0 : nsub);
                 st0 += kDepth) {
                float l[kDepth][E], qv[kDepth][E];
                bool have[kDepth];
#pragma unroll
                for (int k = 0; k < kDepth; ++k)
                    have[k] = st0 + k < nsub && load_unit(st0 + k, l[k], qv[k]);
#pragma unroll
                for (int k = 0; k < kDepth; ++k) {
                    const int64_t st = st0 + k;
                    if (st >= nsub)
                        break;
                    float w[E];
                    if (have[k])
                        cpart += unit_weights(l[k], qv[k], w, badq);
                    if (++gcnt == g32 || st + 1 == nsub) {  // chunk `chunk` ends here
                        const float ct = warp_sum(cpart);
                        cpart = 0.f;
                        if (lane == 0)
                            ctot[warp][chunk] = ct;
                        ++chunk;
                        gcnt = 0;
                        acc_add(wt, wtc, ct);
                    }
                }
            }
            wt -= wtc;
            const int s3 = exchange(make_float4(wt, __any_sync(kFull, badq) ? 1.f : 0.f, 0.f, 0.f));
            if (s3 < 0) {
                state = SV_ERR_TIMEOUT;
                break;
            }
            // totals in vocabulary order: CTA rank, then warp
            float bq = 0.f;
            for (int p = lane; p < P; p += 32)
                bq = fmaxf(bq, part[s3][p].y);
            if (__any_sync(kFull, bq != 0.f)) {
                state = SV_ERR_NONFINITE;
                break;
            }
            Sw = 0.f;
            for (int p = 0; p < P; ++p)
                Sw += part[s3][p].x;
            if (Sw > 0.f || fallback)
                break;
            fallback = true;  // residual all zero: draw from p~_j itself
        }
        if (state == SV_OK) {
            const int s3 = (int)((xcnt - 1) & 1u);
            t = us[K] * Sw;
            float cum = 0.f;
            int last_pos = -1;
            for (int p = 0; p < P; ++p) {
                const float w = part[s3][p].x;
                if (w > 0.f)
                    last_pos = p;
                if (owner < 0 && cum + w > t) {
                    owner = p;
                    cum_before = cum;
                }
                cum += w;
            }
            if (owner < 0) {  // rounding left the point past the last positive total
                owner = last_pos;
                cum_before = 0.f;
                for (int p = 0; p < last_pos; ++p)
                    cum_before += part[s3][p].x;
            }
        }
        // ---- the owner warp locates the token and writes the outputs ----
        if (state == SV_OK && owner == rank * kNW + warp) {
            const float tl = t - cum_before;
            int64_t tok = -1;
            if (listed) {
                // first survivor whose running weight passes the point, or
                // (rounding) the last one with weight
                float run = 0.f;
                int pick = -1, lastk = -1;
                for (int k0 = 0; k0 < ncl && pick < 0; k0 += 32) {
                    const int k = k0 + lane;
                    const float w = k < ncl ? cl_v[k] : 0.f;
                    float inc = w;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float v = __shfl_up_sync(kFull, inc, o);
                        if (lane >= o)
                            inc += v;
                    }
                    const unsigned pos = __ballot_sync(kFull, w > 0.f);
                    if (pos)
                        lastk = k0 + 31 - __clz(pos);
                    const unsigned hit = __ballot_sync(kFull, w > 0.f && run + inc > tl);
                    if (hit)
                        pick = k0 + __ffs(hit) - 1;
                    run += __shfl_sync(kFull, inc, 31);
                }
                if (pick < 0)
                    pick = lastk;
                tok = pick >= 0 ? sv_i[pick] : 0;
            } else {
                // the chunk holding the crossing point (same sums as the total)
                int fc = -1, lastc = -1;
                float before = 0.f, lastc_before = 0.f;
                {
                    float run = 0.f, rc = 0.f;
                    for (int ch = 0; ch < nch; ++ch) {
                        const float x = ctot[warp][ch];
                        const float cur = run - rc;
                        if (x > 0.f) {
                            lastc = ch;
                            lastc_before = cur;
                        }
                        if (cur + x > tl) {
                            fc = ch;
                            before = cur;
                            break;
                        }
                        acc_add(run, rc, x);
                    }
                }
                if (fc < 0) {  // rounding: the last chunk with weight
                    fc = lastc;
                    before = lastc_before;
                }
                float run = before;
                int64_t last = -1;
                const int64_t s_end = min(nsub, (int64_t)(fc + 1) * g);
                for (int64_t st = (int64_t)fc * g; st < s_end && tok < 0; ++st) {
                    float l[E], qv[E], w[E];
                    bool dummy = false;
                    float lt = 0.f;
    #pragma unroll
                    for (int k = 0; k < E; ++k)
                        w[k] = 0.f;
                    const int64_t ui = w0 + st * 32 + lane;
                    if (load_unit(st, l, qv))
                        lt = unit_weights(l, qv, w, dummy);
                    int lpos = -1;
                    for (int k = 0; k < U; ++k)
                        if (w[k] > 0.f)
                            lpos = k;
                    const long long mylast = lpos >= 0 ? (long long)(ui * U + lpos) : -1ll;
                    long long wl_last = mylast;
    #pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        const long long ov = __shfl_xor_sync(kFull, wl_last, o);
                        wl_last = wl_last > ov ? wl_last : ov;
                    }
                    if (wl_last > last)
                        last = wl_last;
                    float inc = lt;  // inclusive scan of the lane sums
    #pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float v = __shfl_up_sync(kFull, inc, o);
                        if (lane >= o)
                            inc += v;
                    }
                    const unsigned hit = __ballot_sync(kFull, run + inc > tl);
                    if (hit) {
                        const int src = __ffs(hit) - 1;
                        long long pick = -1;
                        if (lane == src) {
                            float acc = run + inc - lt;
                            for (int k = 0; k < U; ++k) {
                                acc += w[k];
                                if (acc > tl && w[k] > 0.f) {
                                    pick = ui * U + k;
                                    break;
                                }
                            }
                            if (pick < 0)  // the crossing fell on this lane's last weight
                                pick = mylast;
                        }
                        tok = __shfl_sync(kFull, pick, src);
                    }
                    run += __shfl_sync(kFull, inc, 31);
                }
                if (tok < 0)
                    tok = last;
            }
            const int32_t token = (int32_t)(v0 + tok);
            for (int i = lane; i <= K; i += 32) {
                a.out_tokens[row0 + i] = i < j ? xs[i] : (i == j ? token : -1);
                if (i < K)
                    a.accept_mask[(int64_t)b * K + i] = i < j ? 1 : 0;
                if (a.row_stats) {
                    a.row_stats[(row0 + i) * 2] = i <= j ? rsm[i] : NAN;
                    a.row_stats[(row0 + i) * 2 + 1] = i <= j ? rss[i] : NAN;
                }
                if (i < K && a.p_draft)
                    a.p_draft[(int64_t)b * K + i] = i <= j ? pdr[i] : NAN;
            }
            if (lane == 0) {
                a.accept_len[b] = j + 1;
                if (a.status)
                    a.status[b] = SV_OK;
                if (a.al_hist)
                    atomicAdd(a.al_hist + j + 1, 1u);
            }
        }
    }

    // ---- a sequence error: rank 0 reports it ----
    if (state != SV_OK && rank == 0 && warp == 0) {
        for (int i = lane; i <= K; i += 32) {
            a.out_tokens[row0 + i] = -1;
            if (i < K)
                a.accept_mask[(int64_t)b * K + i] = 0;
            if (a.row_stats) {
                a.row_stats[(row0 + i) * 2] = NAN;
                a.row_stats[(row0 + i) * 2 + 1] = NAN;
            }
            if (i < K && a.p_draft)
                a.p_draft[(int64_t)b * K + i] = NAN;
        }
        if (lane == 0) {
            a.accept_len[b] = 0;
            if (a.status)
                a.status[b] = state;
            atomicOr(a.err_word, 1u << state);
            if (a.al_hist)
                atomicAdd(a.al_hist, 1u);
        }
    }
    // no CTA leaves while a push into it may still be on its way
    if (!ready)
        cluster_wait();
    cluster_arrive();
    cluster_wait();
}

}  // namespace

namespace sv {

int trunc_launch(const TruncLaunch& g, void* stream) {
    TArgs a;
    std::memset(&a, 0, sizeof a);
    a.logits = g.logits;
    a.q = g.q;
    a.tokens = g.tokens;
    a.u = g.u;
    a.accept_len = g.accept_len;
    a.out_tokens = g.out_tokens;
    a.accept_mask = g.accept_mask;
    a.row_stats = g.row_stats;
    a.p_draft = g.p_draft;
    a.status = g.status;
    a.err_word = g.err_word;
    a.al_hist = g.al_hist;
    a.V = g.V;
    a.slice = g.slice;
    a.B = g.B;
    a.K = g.K;
    a.C = g.C;
    a.vec = g.vec;
    a.qvec = g.qvec;
    a.dlogits = g.dlogits;
    a.c = g.c;
    a.cd = g.cd;
    a.T = g.T;
    a.dmin = g.dmin;
    a.top_p = g.top_p;
    a.wait_ns = g.wait_ns;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)((int64_t)g.B * g.C), 1, 1);
    cfg.blockDim = dim3(kNT, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)g.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // q given, or draft logits (with a filter on: the untruncated draft-logit
    // verify runs on the sampled verify's kernel)
    cudaError_t e;
    if (!g.dlogits)
        e = g.es == 2 ? cudaLaunchKernelEx(&cfg, sv_trunc_kernel<2, false>, a)
                      : cudaLaunchKernelEx(&cfg, sv_trunc_kernel<4, false>, a);
    else
        e = g.es == 2 ? cudaLaunchKernelEx(&cfg, sv_trunc_kernel<2, true>, a)
                      : cudaLaunchKernelEx(&cfg, sv_trunc_kernel<4, true>, a);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return 0;
}

}  // namespace sv
