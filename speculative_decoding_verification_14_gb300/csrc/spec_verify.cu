// spec_verify.cu -- batched speculative-decoding verification for GB300 (sm_103a).
//
// Method (pages cited by title and section):
//  [P1] reactapp.top, "Speculative decoding and early exit: speeding up
//       autoregressive decode", section "Speculative decoding: draft first,
//       then verify": p_i = softmax(row_i / T); test the drafts in order; stop
//       at the first rejection; draw the replacement from relu(p - q)
//       normalised; when all K pass, draw a bonus token from row K.
//  [P2] trefon.com, "Decode is memory-bound: a ~59 tok/s ceiling on an RTX
//       4090 and how speculative decoding breaks it", section "Speculative
//       decoding": keep x with probability min(1, p(x)/q(x)).
//  [P3] agentnet.co.il, "New technical post reveals how speculative decoding
//       speeds up LLM inference without hurting accuracy", section "How it
//       works in practice": accepted length in [1, 1 + D].
//
// Design (one launch per call, no global workspace besides a 4-byte error word):
//  * one thread-block cluster of C CTAs per sequence; CTA r owns a contiguous
//    vocabulary slice of every row of that sequence;
//  * a row slice moves HBM -> shared memory with one cp.async.bulk (the TMA
//    bulk-copy engine) completing on an mbarrier; each warp reduces the
//    vectors it owns to a (max, sum of exponentials) pair with packed f32x2
//    arithmetic and publishes it -- no CTA-wide barrier inside a row step;
//  * after one cluster barrier, warp 0 of every CTA reads the C x warps
//    partial pairs through distributed shared memory and merges them in a
//    fixed order in double precision, so every CTA reaches the same
//    accept/reject decision without a broadcast;
//  * rows are consumed in order and the loop stops at the first rejection,
//    like the pages' loop, so rows after it are never read;
//  * the residual (or bonus) draw is split across the cluster: the rejected
//    draft row is bulk-prefetched into L2 as soon as the rejection is known,
//    each CTA weighs its slice (logits still in shared memory), per-warp scans
//    give tile and warp totals, the per-CTA totals meet in distributed shared
//    memory, and the crossing is located by warp-parallel scans down to one
//    entry in the owning CTA.
#include <cuda_runtime.h>
#include <cooperative_groups.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace {

using sv::kMaxK;
using sv::kMaxRows;

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxWarps = 16;
constexpr int kStateRun = 0, kStateSample = 1, kStateError = 2;
constexpr int kModeResidual = 0, kModeBonus = 1, kModeTargetRow = 2;

struct SvArgs {
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
    int64_t V;
    int64_t slice;
    int B, K, C, G;
    int rowbuf_bytes;
    int part_offset;        // bytes from the fixed state to the per-warp partials
    int wt_offset;          // bytes from the fixed state to the tile/warp totals
    int bulk;
    int qvec;
    int prefetch_next;      // 1: L2-prefetch the next row slice while this one is processed
    float c_hi, c_lo;       // log2(e)/T = c_hi + c_lo with c_lo > 0
    float T;
    unsigned long long wait_ns;
};

// Fixed shared state of one CTA.  samp_* is read by the other CTAs of the
// cluster through distributed shared memory (so are the per-warp partials,
// which live after this struct).
struct FF {  // hi + lo, see the double-float helpers below
    float hi, lo;
};

struct __align__(16) SvShared {
    unsigned long long mbar;
    FF samp_tot[2];
    int samp_bad[2];
    FF wtot[kMaxWarps];
    int x[kMaxK];
    float u[kMaxRows];
    float lx[kMaxK];
    float qx[kMaxK];
    float rs_m[kMaxRows];
    float rs_s[kMaxRows];
    float pd[kMaxK];
    int state, j, code, ndec, mode, tok, owner, take_last, loc_tile, loc_warp;
    float rowM;
    FF rowS, loc_rem;
};
static_assert(sizeof(SvShared) + 64 <= sv::kFixedSmem, "fixed shared state outgrew its reservation");

// ------------------------------------------------------------------ PTX -----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bulk copy global -> own shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk prefetch of a global range into L2 (no destination, no completion).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
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

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar`, giving up after `limit_ns` (and after a
// fixed number of polls, whichever comes first).  Returns false on give-up.
__device__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0 && global_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that returns NaN when either input is NaN (IEEE maxNum would drop it)
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^((l - m) * log2(e)/T) for a pair of entries.  The exponent is formed as
// d*c_hi + d*c_lo with d = l - m (exact for bf16 inputs), so the only
// roundings are the final one and the ex2 approximation.  c_lo > 0 keeps a
// -inf entry at -inf (-inf*c_lo = -inf), so it weighs exactly 0.
__device__ __forceinline__ float2 exp2_pair(float2 l, float2 neg_m, float2 chi, float2 clo) {
    const float2 d = __fadd2_rn(l, neg_m);
    const float2 y = __ffma2_rn(d, chi, __fmul2_rn(d, clo));
    return make_float2(ex2_approx(y.x), ex2_approx(y.y));
}

// ------------------------------------------ double-float (fp32 pairs) -----
// A value hi + lo with |lo| <= ulp(hi)/2, built from exact fp32
// transformations (two-sum, two-product): about 44 significant bits, enough
// for every running total and threshold here, all on the FP32 pipe (GB300's
// FP64 units are far too slow to use per row).

__device__ __forceinline__ FF two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}

__device__ __forceinline__ FF fast_two_sum(float a, float b) {  // needs |a| >= |b| or a == 0
    const float s = a + b;
    return {s, b - (s - a)};
}

__device__ __forceinline__ FF two_prod(float a, float b) {
    const float p = a * b;
    return {p, fmaf(a, b, -p)};
}

__device__ __forceinline__ FF ff_add(FF x, FF y) {
    FF t = two_sum(x.hi, y.hi);
    t.lo += x.lo + y.lo;
    return fast_two_sum(t.hi, t.lo);
}

__device__ __forceinline__ FF ff_add(FF x, float y) {
    FF t = two_sum(x.hi, y);
    t.lo += x.lo;
    return fast_two_sum(t.hi, t.lo);
}

__device__ __forceinline__ FF ff_neg(FF x) { return {-x.hi, -x.lo}; }

__device__ __forceinline__ FF ff_mul(FF x, FF y) {
    FF p = two_prod(x.hi, y.hi);
    p.lo = fmaf(x.hi, y.lo, fmaf(x.lo, y.hi, p.lo));
    return fast_two_sum(p.hi, p.lo);
}

// x > y for double-float values
__device__ __forceinline__ bool ff_gt(FF x, FF y) {
    const FF d = ff_add(x, ff_neg(y));
    return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

__device__ __forceinline__ FF shfl_ff(FF v, int src) {
    return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

__device__ __forceinline__ FF shfl_up_ff(FF v, int d) {
    return {__shfl_up_sync(0xffffffffu, v.hi, d), __shfl_up_sync(0xffffffffu, v.lo, d)};
}

__device__ __forceinline__ FF shfl_down_ff(FF v, int d) {
    return {__shfl_down_sync(0xffffffffu, v.hi, d), __shfl_down_sync(0xffffffffu, v.lo, d)};
}

// (l - m) * log2(e)/T as hi + lo, with the difference and the product formed
// exactly (two-sum, two-product).  Needs finite l and m.
__device__ __forceinline__ FF exp2_arg_ff(float l, float m, float c_hi, float c_lo) {
    const FF d = two_sum(l, -m);
    FF p = two_prod(d.hi, c_hi);
    p.lo = fmaf(d.hi, c_lo, fmaf(d.lo, c_hi, p.lo));
    return fast_two_sum(p.hi, p.lo);
}

// 2^y for y = hi + lo <= 0 to about one ulp, on the FMA pipe (used for the
// few values that must be accurate: merge weights and p(x)).  y = n + f with
// n = rint(hi) and |f| <= 1/2 (lo folded into f); 2^f = e^(f ln 2) by its
// Taylor series to degree 7 in (f ln 2), whose truncation error on that
// interval is below 1e-8 relative; 2^n is applied with ldexpf.
__device__ __forceinline__ float exp2_accurate(FF y) {
    if (!(y.hi > -160.f))
        return 0.f;
    const float n = rintf(y.hi);
    const float f = (y.hi - n) + y.lo;
    // coefficients (ln 2)^k / k!, k = 7 .. 0
    float p = 1.5252733804059840e-05f;
    p = fmaf(p, f, 1.5403530393381606e-04f);
    p = fmaf(p, f, 1.3333558146428443e-03f);
    p = fmaf(p, f, 9.6181291076284772e-03f);
    p = fmaf(p, f, 5.5504108664821580e-02f);
    p = fmaf(p, f, 2.4022650695910071e-01f);
    p = fmaf(p, f, 6.9314718055994531e-01f);
    p = fmaf(p, f, 1.0f);
    return ldexpf(p, (int)n);
}

// 2^((l - m) log2e/T) accurately; 0 for l = -inf.
__device__ __forceinline__ float exp2_diff_accurate(float l, float m, float c_hi, float c_lo) {
    if (!(l > -INFINITY))
        return 0.f;
    return exp2_accurate(exp2_arg_ff(l, m, c_hi, c_lo));
}

// ------------------------------------------------------------ elements -----

template <int ES>
struct Elem;
template <>
struct Elem<4> {
    static constexpr int E = 4;  // entries per 16-byte vector
    static constexpr uint32_t kNegInf = 0xff800000u;
    __device__ static __forceinline__ void unpack(const uint4 w, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        f[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
    __device__ static __forceinline__ float load(const void* base, int64_t idx) {
        return __ldg(static_cast<const float*>(base) + idx);
    }
    __device__ static __forceinline__ void store_raw(unsigned char* buf, int64_t k, uint32_t bits) {
        reinterpret_cast<uint32_t*>(buf)[k] = bits;
    }
    __device__ static __forceinline__ uint32_t load_raw(const void* base, int64_t idx) {
        return __ldg(static_cast<const uint32_t*>(base) + idx);
    }
    __device__ static __forceinline__ float vec_max(const uint4 w, float m) {
        return fmax_nan(m, fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                                    fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w))));
    }
};
template <>
struct Elem<2> {
    static constexpr int E = 8;
    static constexpr uint32_t kNegInf = 0xff80u;
    __device__ static __forceinline__ void unpack(const uint4 w, float2 (&f)[4]) {
        f[0] = make_float2(bf16_lo(w.x), bf16_hi(w.x));
        f[1] = make_float2(bf16_lo(w.y), bf16_hi(w.y));
        f[2] = make_float2(bf16_lo(w.z), bf16_hi(w.z));
        f[3] = make_float2(bf16_lo(w.w), bf16_hi(w.w));
    }
    __device__ static __forceinline__ float load(const void* base, int64_t idx) {
        const unsigned short h = __ldg(static_cast<const unsigned short*>(base) + idx);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ static __forceinline__ void store_raw(unsigned char* buf, int64_t k, uint32_t bits) {
        reinterpret_cast<unsigned short*>(buf)[k] = static_cast<unsigned short>(bits);
    }
    __device__ static __forceinline__ uint32_t load_raw(const void* base, int64_t idx) {
        return __ldg(static_cast<const unsigned short*>(base) + idx);
    }
};

// ------------------------------------------------------- warp helpers -----

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Sum over the warp, result in every lane (reduced in one fixed order, then
// broadcast from lane 0 so that all lanes hold the same bits).
__device__ __forceinline__ float warp_sum_bcast(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_down_sync(kFull, v, o);
    return __shfl_sync(kFull, v, 0);
}

__device__ __forceinline__ FF warp_sum_bcast(FF v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = ff_add(v, shfl_down_ff(v, o));
    return shfl_ff(v, 0);
}

__device__ __forceinline__ float warp_incl_scan(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(kFull, v, o);
        if (lane >= o)
            v += n;
    }
    return v;
}

__device__ __forceinline__ FF warp_incl_scan(FF v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const FF n = shfl_up_ff(v, o);
        if (lane >= o)
            v = ff_add(v, n);
    }
    return v;
}

// Exclusive prefix from an inclusive scan: the previous lane's value, `first` in lane 0.
__device__ __forceinline__ FF warp_excl_from_incl(FF incl, FF first) {
    const FF prev = shfl_up_ff(incl, 1);
    return (threadIdx.x & 31) ? prev : first;
}

// First lane whose inclusive running total exceeds `rem`; when none does (a
// rounding corner), the last lane with a positive part and take_last = 1.
// Lanes beyond `n` must hold part = 0.  Returns -1 only if every part is 0.
__device__ __forceinline__ int pick_lane(float part, FF incl, FF rem, int n, int& take_last) {
    const int lane = threadIdx.x & 31;
    const unsigned cross = __ballot_sync(kFull, lane < n && !take_last && ff_gt(incl, rem));
    if (cross)
        return __ffs(cross) - 1;
    const unsigned pos = __ballot_sync(kFull, lane < n && part > 0.f);
    take_last = 1;
    return pos ? 31 - __clz(pos) : -1;
}

// Per-warp (max, sum of exponentials relative to that max) over the vectors of
// one staged row slice this warp owns (vectors warp*32 + lane + k*NT).  The
// same value is returned in every lane.
template <int ES, int NT>
__device__ __forceinline__ float2 warp_slice_stats(const unsigned char* buf, int nvec, float c_hi,
                                                   float c_lo) {
    constexpr int E = Elem<ES>::E;
    const int tid = threadIdx.x;
    const uint4* vbuf = reinterpret_cast<const uint4*>(buf);
    float m;
    if constexpr (ES == 2) {
        uint32_t acc = 0xff80ff80u;
        for (int vi = tid; vi < nvec; vi += NT) {
            const uint4 w = vbuf[vi];
            acc = bf16x2_max_nan(bf16x2_max_nan(acc, w.x), bf16x2_max_nan(w.y, w.z));
            acc = bf16x2_max_nan(acc, w.w);
        }
        m = fmax_nan(bf16_lo(acc), bf16_hi(acc));
    } else {
        m = -INFINITY;
        for (int vi = tid; vi < nvec; vi += NT)
            m = Elem<4>::vec_max(vbuf[vi], m);
    }
    m = warp_max_nan(m);
    float s = 0.f;
    if (m > -INFINITY && m < INFINITY) {  // uniform within the warp
        const float2 neg_m = make_float2(-m, -m), chi = make_float2(c_hi, c_hi),
                     clo = make_float2(c_lo, c_lo);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        for (int vi = tid; vi < nvec; vi += NT) {
            float2 f[E / 2];
            Elem<ES>::unpack(vbuf[vi], f);
#pragma unroll
            for (int k = 0; k < E / 2; k += 2) {
                a0 = __fadd2_rn(a0, exp2_pair(f[k], neg_m, chi, clo));
                a1 = __fadd2_rn(a1, exp2_pair(f[k + 1], neg_m, chi, clo));
            }
        }
        s = warp_sum_bcast((a0.x + a0.y) + (a1.x + a1.y));
    }
    return make_float2(m, s);
}

// Draft probabilities for one 16-byte vector of the slice (E entries); entries
// at or past L read as 0.
template <int ES>
__device__ __forceinline__ void load_q_vec(const float* qrow, int vi, int64_t L, int qvec,
                                           float (&qq)[Elem<ES>::E]) {
    constexpr int E = Elem<ES>::E;
    const int64_t base = (int64_t)vi * E;
    if (qvec && base + E <= L) {
#pragma unroll
        for (int k = 0; k < E; k += 4) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(qrow + base + k));
            qq[k] = t.x;
            qq[k + 1] = t.y;
            qq[k + 2] = t.z;
            qq[k + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < E; ++k)
            qq[k] = base + k < L ? __ldg(qrow + base + k) : 0.f;
    }
}

// Draw weights of one vector: residual max(0, p - q) (mode 0) or the
// unnormalised target weights exp(z - max) (modes 1 and 2).  Entries at or
// past L weigh 0.  `bad` is raised by a NaN, infinite or negative q value.
template <int ES>
__device__ __forceinline__ float vec_weights(const unsigned char* buf, int vi, int64_t L,
                                             const float (&qq)[Elem<ES>::E], int mode, float M,
                                             float c_hi, float c_lo, float inv_s,
                                             float (&w)[Elem<ES>::E], bool& bad) {
    constexpr int E = Elem<ES>::E;
    float2 f[E / 2];
    Elem<ES>::unpack(reinterpret_cast<const uint4*>(buf)[vi], f);
    const float2 neg_m = make_float2(-M, -M), chi = make_float2(c_hi, c_hi),
                 clo = make_float2(c_lo, c_lo);
    const int64_t base = (int64_t)vi * E;
    float ts = 0.f;
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        const float2 e = exp2_pair(f[k], neg_m, chi, clo);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int idx = 2 * k + h;
            const float ev = h ? e.y : e.x;
            float wk;
            if (mode == kModeResidual) {
                const float qv = qq[idx];
                if (base + idx < L && !(qv >= 0.f && qv < INFINITY))
                    bad = true;
                wk = fmaxf(__fmaf_rn(ev, inv_s, -qv), 0.f);
            } else {
                wk = ev;
            }
            w[idx] = base + idx < L ? wk : 0.f;
            ts += w[idx];
        }
    }
    return ts;
}

// --------------------------------------------------------------- kernel -----

// Residency target: 1536 threads per SM (registers capped accordingly).
template <int ES, int NT>
__global__ void __launch_bounds__(NT, 1536 / NT) sv_verify_kernel(const __grid_constant__ SvArgs a) {
    constexpr int E = Elem<ES>::E;
    constexpr int NW = NT / 32;
    static_assert(NW <= kMaxWarps, "too many warps");
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)a.C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K;
    const int64_t V = a.V;
    const int C = a.C;
    const int G = a.G;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* bufs = smem_raw;
    unsigned char* fixed = smem_raw + (size_t)G * a.rowbuf_bytes;
    SvShared& sh = *reinterpret_cast<SvShared*>(fixed);
    float2* part = reinterpret_cast<float2*>(fixed + a.part_offset);  // [2][G][NW] (max, sum)
    int* part_flag = reinterpret_cast<int*>(part + 2 * G * NW);       // [2][NW]
    float* wt = reinterpret_cast<float*>(fixed + a.wt_offset);          // [tiles][NW]

    // this CTA's vocabulary slice
    const int64_t v0 = (int64_t)rank * a.slice;
    const int64_t L = v0 < V ? (V - v0 < a.slice ? V - v0 : a.slice) : 0;
    const int nvec = (int)((L + E - 1) / E);
    const int64_t row0 = (int64_t)b * (K + 1);  // first logits row of this sequence

    if (tid == 0) {
        mbar_init(&sh.mbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    uint32_t phase = 0;
    bool timed_out = false;  // per thread; published per warp

    auto row_src = [&](int row) {
        return static_cast<const unsigned char*>(a.logits) + ((row0 + row) * V + v0) * ES;
    };
    // Moves rows g0 .. g0+ng-1 of this sequence's slice into shared memory.
    auto load_group = [&](int g0, int ng) {
        if (L == 0)
            return;
        if (a.bulk) {
            if (tid == 0) {
                fence_proxy_async();
                const uint32_t bytes = (uint32_t)(L * ES);
                mbar_arrive_expect_tx(&sh.mbar, bytes * (uint32_t)ng);
                for (int r = 0; r < ng; ++r)
                    bulk_copy_g2s(bufs + (size_t)r * a.rowbuf_bytes, row_src(g0 + r), bytes,
                                  &sh.mbar);
                if (a.prefetch_next)
                    for (int r = g0 + ng; r < g0 + 2 * ng && r <= K; ++r)
                        bulk_prefetch_l2(row_src(r), bytes);
            }
        } else {
            const int64_t lpad = (int64_t)nvec * E;
            for (int r = 0; r < ng; ++r) {
                unsigned char* dst = bufs + (size_t)r * a.rowbuf_bytes;
                const int64_t gbase = (row0 + g0 + r) * V + v0;
                for (int64_t k = tid; k < lpad; k += NT)
                    Elem<ES>::store_raw(dst, k,
                                        k < L ? Elem<ES>::load_raw(a.logits, gbase + k)
                                              : Elem<ES>::kNegInf);
            }
        }
    };
    auto wait_group = [&]() {
        if (L == 0)
            return;
        if (a.bulk) {
            if (!mbar_wait_bounded(&sh.mbar, phase, a.wait_ns))
                timed_out = true;
            phase ^= 1u;
        } else {
            __syncthreads();
        }
    };

    // first group's copy goes out before anything else
    load_group(0, G < K + 1 ? G : K + 1);

    // per-sequence inputs: drafts, uniforms, and the gathered p/q inputs at the drafts
    if (tid < K)
        sh.x[tid] = a.tokens[(int64_t)b * K + tid];
    if (tid <= K)
        sh.u[tid] = a.u[(int64_t)b * (K + 1) + tid];
    __syncthreads();
    if (tid == 0) {
        int code = SV_OK;
        for (int i = 0; i < K && code == SV_OK; ++i)
            if (sh.x[i] < 0 || (int64_t)sh.x[i] >= V)
                code = SV_ERR_TOKEN_RANGE;
        for (int i = 0; i <= K && code == SV_OK; ++i)
            if (!(sh.u[i] >= 0.f && sh.u[i] < 1.f))
                code = SV_ERR_UNIFORM_RANGE;
        sh.code = code;
        sh.state = code == SV_OK ? kStateRun : kStateError;
        sh.ndec = 0;
        sh.j = -1;
    }
    __syncthreads();
    if (sh.state == kStateRun && tid < K) {
        const int x = sh.x[tid];
        sh.lx[tid] = Elem<ES>::load(a.logits, (row0 + tid) * V + x);
        sh.qx[tid] = __ldg(a.q + ((int64_t)b * K + tid) * V + x);
    }
    // (made visible to warp 0 by the cluster barrier below)

    // ---- test loop over groups of rows, in order ([P1]) ----
    int par = 0;
    int g0 = 0;
    int gcur = 0;  // first row of the group currently staged
    for (;;) {
        const int ng = G < K + 1 - g0 ? G : K + 1 - g0;
        wait_group();
        gcur = g0;
        if (sh.state != kStateRun)
            break;
        for (int r = 0; r < ng; ++r) {
            const float2 ms = L ? warp_slice_stats<ES, NT>(bufs + (size_t)r * a.rowbuf_bytes, nvec,
                                                           a.c_hi, a.c_lo)
                                : make_float2(-INFINITY, 0.f);
            if (lane == 0)
                part[(par * G + r) * NW + warp] = ms;
        }
        {
            const int anyto = __any_sync(kFull, timed_out);
            if (lane == 0)
                part_flag[par * NW + warp] = anyto;
        }
        cluster.sync();

        // combine the C * NW partial pairs of each row in a fixed order, then decide
        if (warp == 0) {
            constexpr int kPer = sv::kMaxCluster * NW / 32;  // partials per lane, at most
            const int P = C * NW;
            int anyflag = 0;
            for (int p = lane; p < P; p += 32)
                anyflag |= cluster.map_shared_rank(part_flag, p / NW)[par * NW + (p % NW)];
            anyflag = __any_sync(kFull, anyflag != 0);
            for (int r = 0; r < ng; ++r) {
                float2 pv[kPer];
                float mloc = -INFINITY;
#pragma unroll
                for (int t = 0; t < kPer; ++t) {
                    const int p = lane + 32 * t;
                    pv[t] = make_float2(-INFINITY, 0.f);
                    if (p < P) {
                        pv[t] = cluster.map_shared_rank(part, p / NW)[(par * G + r) * NW + (p % NW)];
                        mloc = fmax_nan(mloc, pv[t].x);
                    }
                }
                const float M = warp_max_nan(mloc);
                const bool finite = M > -INFINITY && M < INFINITY;
                FF acc = {0.f, 0.f};
                if (finite) {
#pragma unroll
                    for (int t = 0; t < kPer; ++t)
                        if (pv[t].y > 0.f)
                            acc = ff_add(acc, two_prod(pv[t].y, exp2_diff_accurate(
                                                                    pv[t].x, M, a.c_hi, a.c_lo)));
                }
                const FF S = warp_sum_bcast(acc);
                // p(x) numerator 2^((l_x - M) log2e/T), on a lane of its own
                float num = 0.f;
                if (lane == 1 && finite && g0 + r < K)
                    num = exp2_diff_accurate(sh.lx[g0 + r], M, a.c_hi, a.c_lo);
                num = __shfl_sync(kFull, num, 1);
                if (lane == 0 && sh.state == kStateRun) {
                    const int i = g0 + r;
                    if (anyflag) {
                        sh.state = kStateError;
                        sh.code = SV_ERR_TIMEOUT;
                    } else if (!finite) {
                        sh.state = kStateError;
                        sh.code = SV_ERR_NONFINITE;
                    } else {
                        const float Sf = S.hi;
                        sh.rs_m[i] = __fdiv_rn(M, a.T);
                        sh.rs_s[i] = Sf;
                        sh.ndec = i + 1;
                        if (i < K) {
                            const float qxf = sh.qx[i];
                            if (!(qxf >= 0.f && qxf < INFINITY)) {
                                sh.state = kStateError;
                                sh.code = SV_ERR_NONFINITE;
                            } else {
                                sh.pd[i] = __fdiv_rn(num, Sf);
                                // u < p(x)/q(x) as u * q(x) * S < 2^((l_x - M) log2e/T):
                                // products only, in double-float
                                const FF lhs = ff_mul(two_prod(sh.u[i], qxf), S);
                                if (!ff_gt(FF{num, 0.f}, lhs)) {
                                    sh.state = kStateSample;
                                    sh.j = i;
                                    sh.mode = kModeResidual;
                                    sh.rowM = M;
                                    sh.rowS = S;
                                    // the draft row is needed now: start pulling it into L2
                                    if (a.qvec && L > 0)
                                        bulk_prefetch_l2(a.q + ((int64_t)b * K + i) * V + v0,
                                                         (uint32_t)(L * 4));
                                }
                            }
                        } else {
                            sh.state = kStateSample;
                            sh.j = K;
                            sh.mode = kModeBonus;
                            sh.rowM = M;
                            sh.rowS = S;
                        }
                    }
                }
                __syncwarp();
            }
        }
        __syncthreads();
        par ^= 1;
        if (sh.state != kStateRun)
            break;
        g0 += ng;
        load_group(g0, G < K + 1 - g0 ? G : K + 1 - g0);
    }

    // ---- corrected or bonus draw over row j ([P1]) ----
    if (sh.state == kStateSample) {
        const int j = sh.j;
        const unsigned char* buf = bufs + (size_t)(j - gcur) * a.rowbuf_bytes;
        const float* qrow = j < K ? a.q + ((int64_t)b * K + j) * V + v0 : nullptr;
        const float M = sh.rowM;
        const float inv_s = __frcp_rn(sh.rowS.hi);
        const float uK = sh.u[K];
        const int ntiles = (nvec + NT - 1) / NT;
        int mode = sh.mode;
        int sp = 0;
        for (int round = 0; round < 2; ++round) {
            bool bad = false;
            FF wacc = {0.f, 0.f};  // this warp's total over all tiles (meaningful in lane 31)
            for (int k = 0; k < ntiles; k += 2) {
                // two tiles in flight: both q loads go out before either is used
                const int vi0 = k * NT + tid, vi1 = vi0 + NT;
                float q0[E], q1[E], w[E];
#pragma unroll
                for (int e = 0; e < E; ++e)
                    q0[e] = q1[e] = 0.f;
                if (mode == kModeResidual) {
                    if (vi0 < nvec)
                        load_q_vec<ES>(qrow, vi0, L, a.qvec, q0);
                    if (vi1 < nvec)
                        load_q_vec<ES>(qrow, vi1, L, a.qvec, q1);
                }
                const float ts0 = vi0 < nvec ? vec_weights<ES>(buf, vi0, L, q0, mode, M, a.c_hi,
                                                               a.c_lo, inv_s, w, bad)
                                             : 0.f;
                const float ts1 = vi1 < nvec ? vec_weights<ES>(buf, vi1, L, q1, mode, M, a.c_hi,
                                                               a.c_lo, inv_s, w, bad)
                                             : 0.f;
                const float in0 = warp_incl_scan(ts0);
                const float in1 = warp_incl_scan(ts1);
                if (lane == 31) {
                    wt[k * NW + warp] = in0;
                    wacc = ff_add(wacc, in0);
                    if (k + 1 < ntiles) {
                        wt[(k + 1) * NW + warp] = in1;
                        wacc = ff_add(wacc, in1);
                    }
                }
            }
            if (lane == 31)
                sh.wtot[warp] = wacc;
            const int anybad = __syncthreads_or(bad);
            if (tid == 0) {
                FF tot = {0.f, 0.f};
                for (int w2 = 0; w2 < NW; ++w2)
                    tot = ff_add(tot, sh.wtot[w2]);
                sh.samp_tot[sp] = tot;
                sh.samp_bad[sp] = anybad;
            }
            cluster.sync();
            if (warp == 0) {
                FF tot = {0.f, 0.f};
                int cbad = 0;
                if (lane < C) {
                    const SvShared* rs = cluster.map_shared_rank(&sh, lane);
                    tot = rs->samp_tot[sp];
                    cbad = rs->samp_bad[sp];
                }
                cbad = __any_sync(kFull, cbad != 0);
                const FF incl = warp_incl_scan(tot);
                const FF S = shfl_ff(incl, C - 1);
                const FF t = ff_mul(FF{uK, 0.f}, S);
                int take_last = 0;
                const int owner = pick_lane(tot.hi, incl, t, C, take_last);
                const FF excl = shfl_ff(warp_excl_from_incl(incl, FF{0.f, 0.f}), owner < 0 ? 0 : owner);
                if (lane == 0) {
                    if (cbad) {
                        sh.state = kStateError;
                        sh.code = SV_ERR_NONFINITE;
                        sh.mode = -1;
                    } else if (S.hi == 0.f && mode == kModeResidual) {
                        // max(0, p - q) vanished (rounding or an unnormalised q):
                        // draw from p_j itself with the same uniform
                        sh.mode = kModeTargetRow;
                    } else if (owner < 0) {
                        // no positive weight anywhere: unreachable when the row max is finite
                        sh.state = kStateError;
                        sh.code = SV_ERR_NONFINITE;
                        sh.mode = -1;
                    } else {
                        sh.mode = -1;  // done
                        sh.owner = owner;
                        sh.take_last = take_last;
                        sh.loc_rem = ff_add(t, ff_neg(excl));
                    }
                }
            }
            __syncthreads();
            if (sh.mode != kModeTargetRow)
                break;
            mode = kModeTargetRow;
            sp ^= 1;
        }

        if (sh.state == kStateSample && rank == sh.owner) {
            // tile, then warp, by warp-parallel scans over the stored totals
            if (warp == 0) {
                int take_last = sh.take_last;
                const FF rem = sh.loc_rem;
                int kk = -1, klast = -1;
                FF carry = {0.f, 0.f}, carry_last = {0.f, 0.f}, acc_at = {0.f, 0.f};
                for (int c0 = 0; c0 < ntiles && kk < 0; c0 += 32) {
                    const int k = c0 + lane;
                    FF tk = {0.f, 0.f};
                    if (k < ntiles)
                        for (int w2 = 0; w2 < NW; ++w2)
                            tk = ff_add(tk, wt[k * NW + w2]);
                    const FF incl = ff_add(warp_incl_scan(tk), carry);
                    const FF excl = warp_excl_from_incl(incl, carry);
                    int tl = take_last;
                    const int pick = pick_lane(tk.hi, incl, rem, ntiles - c0, tl);
                    if (!tl && pick >= 0) {
                        kk = c0 + pick;
                        acc_at = shfl_ff(excl, pick);
                    } else if (pick >= 0) {
                        klast = c0 + pick;
                        carry_last = shfl_ff(excl, pick);
                    }
                    carry = shfl_ff(incl, 31);
                }
                if (kk < 0) {
                    take_last = 1;
                    kk = klast;
                    acc_at = carry_last;
                }
                float tw = 0.f;
                if (kk >= 0 && lane < NW)
                    tw = wt[kk * NW + lane];
                const FF inclw = ff_add(warp_incl_scan(FF{tw, 0.f}), acc_at);
                const FF exclw = warp_excl_from_incl(inclw, acc_at);
                const int ww = pick_lane(tw, inclw, rem, NW, take_last);
                const FF accw = shfl_ff(exclw, ww < 0 ? 0 : ww);
                if (lane == 0) {
                    sh.loc_tile = kk;
                    sh.loc_warp = ww;
                    sh.take_last = take_last;
                    sh.loc_rem = ff_add(rem, ff_neg(accw));
                }
            }
            __syncthreads();
            if (warp == sh.loc_warp && sh.loc_tile >= 0) {
                // this warp re-derives the same weights and scan, then finds the
                // lane and the entry where the running sum passes the remainder
                int take_last = sh.take_last;
                const FF rem = sh.loc_rem;
                const int vi = sh.loc_tile * NT + tid;
                float qq[E], w[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    qq[e] = 0.f;
                    w[e] = 0.f;
                }
                bool dummy = false;
                float ts = 0.f;
                if (vi < nvec) {
                    if (mode == kModeResidual)
                        load_q_vec<ES>(qrow, vi, L, a.qvec, qq);
                    ts = vec_weights<ES>(buf, vi, L, qq, mode, M, a.c_hi, a.c_lo, inv_s, w, dummy);
                }
                const float incl = warp_incl_scan(ts);
                const int pick = pick_lane(ts, FF{incl, 0.f}, rem, 32, take_last);
                float prev = __shfl_up_sync(kFull, incl, 1);
                if (lane == 0)
                    prev = 0.f;
                const float excl = __shfl_sync(kFull, prev, pick < 0 ? 0 : pick);
                if (lane == pick) {
                    int e_hit = -1, e_last = -1;
                    FF acc = {excl, 0.f};
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if (w[e] > 0.f)
                            e_last = e;
                        acc = ff_add(acc, w[e]);
                        if (e_hit < 0 && !take_last && ff_gt(acc, rem))
                            e_hit = e;
                    }
                    const int e = e_hit >= 0 ? e_hit : e_last;
                    sh.tok = (int)(v0 + (int64_t)vi * E + (e >= 0 ? e : 0));
                }
            }
            __syncthreads();
            // outputs of a finished sequence
            const int tok = sh.tok;
            for (int i = tid; i <= K; i += NT) {
                a.out_tokens[(int64_t)b * (K + 1) + i] = i < j ? sh.x[i] : (i == j ? tok : -1);
                if (i < K)
                    a.accept_mask[(int64_t)b * K + i] = i < j ? 1 : 0;
            }
            if (tid == 0) {
                a.accept_len[b] = j + 1;
                if (a.status)
                    a.status[b] = SV_OK;
            }
        }
    }

    // ---- rank 0 reports the per-row statistics, or the sequence error ----
    if (rank == 0) {
        const bool err = sh.state == kStateError;
        const int ndec = err ? 0 : sh.ndec;
        for (int i = tid; i <= K; i += NT) {
            if (a.row_stats) {
                a.row_stats[((int64_t)b * (K + 1) + i) * 2] = i < ndec ? sh.rs_m[i] : NAN;
                a.row_stats[((int64_t)b * (K + 1) + i) * 2 + 1] = i < ndec ? sh.rs_s[i] : NAN;
            }
            if (i < K && a.p_draft)
                a.p_draft[(int64_t)b * K + i] = i < ndec ? sh.pd[i] : NAN;
            if (err) {
                a.out_tokens[(int64_t)b * (K + 1) + i] = -1;
                if (i < K)
                    a.accept_mask[(int64_t)b * K + i] = 0;
            }
        }
        if (err && tid == 0) {
            a.accept_len[b] = 0;
            if (a.status)
                a.status[b] = sh.code;
            atomicOr(a.err_word, 1u << sh.code);
        }
    }

    // a copy that timed out may still land: give it one more bounded wait
    if (timed_out)
        (void)mbar_wait_bounded(&sh.mbar, phase ^ 1u, a.wait_ns);
    // nobody leaves while a peer may still read its shared memory
    cluster.sync();
}

// ----------------------------------------------------------------- host -----

using KernelFn = void (*)(SvArgs);

KernelFn pick_kernel(int es, int threads) {
    if (es == 2) {
        if (threads == 128) return sv_verify_kernel<2, 128>;
        if (threads == 256) return sv_verify_kernel<2, 256>;
        if (threads == 512) return sv_verify_kernel<2, 512>;
    } else {
        if (threads == 128) return sv_verify_kernel<4, 128>;
        if (threads == 256) return sv_verify_kernel<4, 256>;
        if (threads == 512) return sv_verify_kernel<4, 512>;
    }
    return nullptr;
}

struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            switched = cudaSetDevice(dev) == cudaSuccess;
        }
    }
    ~DeviceGuard() {
        if (switched)
            cudaSetDevice(prev);
    }
};

}  // namespace

struct sv_ctx {
    int device = 0;
    int max_B = 0, max_K = 0;
    int64_t max_V = 0;
    int num_sms = 0, smem_optin = 0, max_cluster = 8;
    uint32_t* d_err = nullptr;
    int ovr_cluster = 0, ovr_group = 0, ovr_threads = 0;
    int ovr_prefetch = -1;  // -1: the planner decides
    unsigned long long wait_ns = 2000000000ull;
    // staging for the host-buffer entry point
    unsigned char* d_stage = nullptr;
    size_t stage_bytes = 0;
};

namespace {

int env_int(const char* name, int dflt) {
    const char* s = std::getenv(name);
    return s && *s ? std::atoi(s) : dflt;
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

int validate(const sv_ctx* ctx, const void* logits, int dtype, const float* q, const int32_t* tokens,
             const float* uniforms, int B, int K, int64_t V, float T, const int32_t* accept_len,
             const int32_t* out_tokens, const uint8_t* accept_mask, const float* row_stats,
             const float* p_draft, const int32_t* status) {
    if (!ctx || !logits || !uniforms || !accept_len || !out_tokens)
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16)
        return SV_ERR_INVALID_ARG;
    if (B < 1 || B > ctx->max_B || K < 0 || K > ctx->max_K || K > kMaxK || V < 1 ||
        V > ctx->max_V)
        return SV_ERR_INVALID_ARG;
    if ((double)B * (double)(K + 1) * (double)V >= 1099511627776.0)  // 2^40
        return SV_ERR_INVALID_ARG;
    if (K > 0 && (!q || !tokens || !accept_mask))
        return SV_ERR_INVALID_ARG;
    if (!(T > 0.f) || !std::isfinite(T))
        return SV_ERR_INVALID_ARG;
    const size_t es = dtype == SV_BF16 ? 2 : 4;
    if (!aligned(logits, es) || (q && !aligned(q, 4)) || (tokens && !aligned(tokens, 4)) ||
        !aligned(uniforms, 4) || !aligned(accept_len, 4) || !aligned(out_tokens, 4) ||
        (row_stats && !aligned(row_stats, 4)) || (p_draft && !aligned(p_draft, 4)) ||
        (status && !aligned(status, 4)))
        return SV_ERR_INVALID_ARG;
    return SV_OK;
}

int make_plan(const sv_ctx* ctx, int B, int K, int64_t V, int dtype, sv_plan* plan) {
    const int rc = spec_verify_plan_for(ctx->num_sms, ctx->smem_optin, ctx->max_cluster, B, K, V,
                                        dtype, ctx->ovr_cluster, ctx->ovr_group, ctx->ovr_threads,
                                        plan);
    if (rc == SV_OK && ctx->ovr_prefetch >= 0)
        plan->prefetch_next = ctx->ovr_prefetch ? 1 : 0;
    return rc;
}

int launch(sv_ctx* ctx, const void* logits, int dtype, const float* q, const int32_t* tokens,
           const float* uniforms, int B, int K, int64_t V, float T, int32_t* accept_len,
           int32_t* out_tokens, uint8_t* accept_mask, float* row_stats, float* p_draft,
           int32_t* status, cudaStream_t stream) {
    sv_plan plan;
    int rc = make_plan(ctx, B, K, V, dtype, &plan);
    if (rc != SV_OK)
        return rc;
    const int es = dtype == SV_BF16 ? 2 : 4;
    KernelFn fn = pick_kernel(es, plan.threads);
    if (!fn)
        return SV_ERR_UNSUPPORTED;

    SvArgs args;
    std::memset(&args, 0, sizeof args);
    args.logits = logits;
    args.q = q;
    args.tokens = tokens;
    args.u = uniforms;
    args.accept_len = accept_len;
    args.out_tokens = out_tokens;
    args.accept_mask = accept_mask;
    args.row_stats = row_stats;
    args.p_draft = p_draft;
    args.status = status;
    args.err_word = ctx->d_err;
    args.V = V;
    args.slice = plan.slice;
    args.B = B;
    args.K = K;
    args.C = plan.cluster;
    args.G = plan.group;
    args.rowbuf_bytes = (int)sv::round_up(plan.slice * es, sv::kRowBufAlign);
    args.part_offset = (int)sv::round_up(sizeof(SvShared), 16);
    args.wt_offset = args.part_offset + (int)sv::partial_bytes(plan.group, plan.threads);
    args.bulk = plan.bulk_copy && aligned(logits, 16) ? 1 : 0;
    args.prefetch_next = plan.prefetch_next && args.bulk ? 1 : 0;
    args.qvec = (V % 4 == 0) && q && aligned(q, 16) ? 1 : 0;
    args.T = T;
    const double c_d = 1.4426950408889634074 / (double)T;  // log2(e) / T
    // c_hi just below c_d so that c_lo = c_d - c_hi is strictly positive: a
    // -inf logit then gives -inf * c_lo = -inf instead of NaN
    args.c_hi = (float)c_d;
    if ((double)args.c_hi >= c_d)
        args.c_hi = std::nextafter(args.c_hi, 0.0f);
    args.c_lo = (float)(c_d - (double)args.c_hi);
    args.wait_ns = ctx->wait_ns;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)plan.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    DeviceGuard guard(ctx->device);
    if (cudaLaunchKernelEx(&cfg, fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

}  // namespace

extern "C" {

int spec_verify_version(void) { return 100; }

const char* spec_verify_strerror(int code) {
    switch (code) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID_ARG: return "invalid argument";
        case SV_ERR_UNSUPPORTED: return "shape not supported by any launch plan";
        case SV_ERR_CUDA: return "CUDA runtime error";
        case SV_ERR_TOKEN_RANGE: return "draft token outside [0, V)";
        case SV_ERR_NONFINITE: return "non-finite target row or invalid draft probability";
        case SV_ERR_TIMEOUT: return "bounded wait for a bulk copy ran out";
        case SV_ERR_UNIFORM_RANGE: return "uniform outside [0, 1)";
        default: return "unknown status";
    }
}

int spec_verify_init(sv_ctx** out, int device, int max_B, int max_K, int64_t max_V) {
    if (!out || max_B < 1 || max_K < 0 || max_K > kMaxK || max_V < 1)
        return SV_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    DeviceGuard guard(device);
    int major = 0, minor = 0, sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    if (major != 10 || minor != 3)  // the kernels are built for sm_103a only
        return SV_ERR_UNSUPPORTED;
    sv_ctx* ctx = new sv_ctx();
    ctx->device = device;
    ctx->max_B = max_B;
    ctx->max_K = max_K;
    ctx->max_V = max_V;
    ctx->num_sms = sms;
    ctx->smem_optin = optin;
    const int ns = env_int("SV_WAIT_MS", 0);
    if (ns > 0)
        ctx->wait_ns = (unsigned long long)ns * 1000000ull;
    int max_cluster = 16;
    const int es_list[2] = {2, 4};
    const int nt_list[3] = {128, 256, 512};
    for (int es : es_list)
        for (int nt : nt_list) {
            KernelFn fn = pick_kernel(es, nt);
            if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin) != cudaSuccess) {
                (void)cudaGetLastError();
                delete ctx;
                return SV_ERR_CUDA;
            }
            if (cudaFuncSetAttribute((const void*)fn,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess) {
                (void)cudaGetLastError();
                max_cluster = 8;
            }
        }
    if (max_cluster == 16) {
        // confirm that a 16-CTA cluster of the widest plan can be resident
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(512, 1, 1);
        cfg.dynamicSmemBytes = 64 * 1024;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, (const void*)pick_kernel(2, 512), &cfg) !=
                cudaSuccess ||
            nclusters < 1) {
            (void)cudaGetLastError();
            max_cluster = 8;
        }
    }
    ctx->max_cluster = max_cluster;
    ctx->ovr_cluster = env_int("SV_CLUSTER", 0);
    ctx->ovr_group = env_int("SV_GROUP", 0);
    ctx->ovr_threads = env_int("SV_THREADS", 0);
    ctx->ovr_prefetch = env_int("SV_PREFETCH", -1);
    if (cudaMalloc(&ctx->d_err, sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(ctx->d_err, 0, sizeof(uint32_t)) != cudaSuccess) {
        (void)cudaGetLastError();
        if (ctx->d_err)
            cudaFree(ctx->d_err);
        delete ctx;
        return SV_ERR_CUDA;
    }
    *out = ctx;
    return SV_OK;
}

int spec_verify_destroy(sv_ctx* ctx) {
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    int rc = SV_OK;
    if (ctx->d_err && cudaFree(ctx->d_err) != cudaSuccess)
        rc = SV_ERR_CUDA;
    if (ctx->d_stage && cudaFree(ctx->d_stage) != cudaSuccess)
        rc = SV_ERR_CUDA;
    delete ctx;
    return rc;
}

int spec_verify_set_plan_override(sv_ctx* ctx, int cluster, int group, int threads) {
    if (!ctx || cluster < 0 || cluster > ctx->max_cluster || group < 0 || group > kMaxRows ||
        (threads != 0 && threads != 128 && threads != 256 && threads != 512))
        return SV_ERR_INVALID_ARG;
    ctx->ovr_cluster = cluster;
    ctx->ovr_group = group;
    ctx->ovr_threads = threads;
    return SV_OK;
}

int spec_verify_get_plan(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype, sv_plan* out) {
    if (!ctx || !out)
        return SV_ERR_INVALID_ARG;
    return make_plan(ctx, B, K, V, logits_dtype, out);
}

int spec_verify_run(sv_ctx* ctx, const void* target_logits, int logits_dtype, const float* q,
                    const int32_t* draft_tokens, const float* uniforms, int B, int K, int64_t V,
                    float temperature, int32_t* accept_len, int32_t* out_tokens,
                    uint8_t* accept_mask, float* row_stats, float* p_draft, int32_t* status,
                    void* stream) {
    const int rc = validate(ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K, V,
                            temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft,
                            status);
    if (rc != SV_OK)
        return rc;
    return launch(ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K, V,
                  temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft, status,
                  static_cast<cudaStream_t>(stream));
}

int spec_verify_get_error(sv_ctx* ctx, void* stream, uint32_t* mask) {
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, ctx->d_err, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ctx->d_err, 0, sizeof(uint32_t), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    if (mask)
        *mask = h;
    for (int code = 1; code < 32; ++code)
        if (h & (1u << code))
            return code;
    return SV_OK;
}

int spec_verify_run_host(sv_ctx* ctx, const void* target_logits, int logits_dtype, const float* q,
                         const int32_t* draft_tokens, const float* uniforms, int B, int K,
                         int64_t V, float temperature, int32_t* accept_len, int32_t* out_tokens,
                         uint8_t* accept_mask, float* row_stats, float* p_draft, int32_t* status,
                         void* stream) {
    int rc = validate(ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K, V,
                      temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft, status);
    if (rc != SV_OK)
        return rc;
    DeviceGuard guard(ctx->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = logits_dtype == SV_BF16 ? 2 : 4;
    auto al = [](size_t n) { return (n + 255) & ~(size_t)255; };
    // staging layout sized to this call; a larger later call replaces it
    const size_t mB = (size_t)B, mK = (size_t)K, mV = (size_t)V;
    const size_t cap_logits = al(mB * (mK + 1) * mV * 4), cap_q = al(mB * mK * mV * 4);
    const size_t cap_tok = al(mB * mK * 4), cap_u = al(mB * (mK + 1) * 4);
    const size_t cap_len = al(mB * 4), cap_out = al(mB * (mK + 1) * 4), cap_mask = al(mB * mK);
    const size_t cap_stats = al(mB * (mK + 1) * 8), cap_pd = al(mB * mK * 4), cap_st = al(mB * 4);
    const size_t need = cap_logits + cap_q + cap_tok + cap_u + cap_len + cap_out + cap_mask +
                        cap_stats + cap_pd + cap_st;
    if (ctx->d_stage && ctx->stage_bytes < need) {
        if (cudaStreamSynchronize(s) != cudaSuccess || cudaFree(ctx->d_stage) != cudaSuccess) {
            (void)cudaGetLastError();
            return SV_ERR_CUDA;
        }
        ctx->d_stage = nullptr;
        ctx->stage_bytes = 0;
    }
    if (!ctx->d_stage) {
        if (cudaMalloc(&ctx->d_stage, need) != cudaSuccess) {
            (void)cudaGetLastError();
            ctx->d_stage = nullptr;
            return SV_ERR_CUDA;
        }
        ctx->stage_bytes = need;
    }
    unsigned char* p = ctx->d_stage;
    void* d_logits = p; p += cap_logits;
    float* d_q = reinterpret_cast<float*>(p); p += cap_q;
    int32_t* d_tok = reinterpret_cast<int32_t*>(p); p += cap_tok;
    float* d_u = reinterpret_cast<float*>(p); p += cap_u;
    int32_t* d_len = reinterpret_cast<int32_t*>(p); p += cap_len;
    int32_t* d_out = reinterpret_cast<int32_t*>(p); p += cap_out;
    uint8_t* d_mask = p; p += cap_mask;
    float* d_stats = reinterpret_cast<float*>(p); p += cap_stats;
    float* d_pd = reinterpret_cast<float*>(p); p += cap_pd;
    int32_t* d_st = reinterpret_cast<int32_t*>(p);

    const size_t nB = (size_t)B, nK = (size_t)K, nV = (size_t)V;
    bool ok = cudaMemcpyAsync(d_logits, target_logits, nB * (nK + 1) * nV * es,
                              cudaMemcpyHostToDevice, s) == cudaSuccess;
    if (K > 0) {
        ok = ok && cudaMemcpyAsync(d_q, q, nB * nK * nV * 4, cudaMemcpyHostToDevice, s) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(d_tok, draft_tokens, nB * nK * 4, cudaMemcpyHostToDevice, s) ==
                       cudaSuccess;
    }
    ok = ok && cudaMemcpyAsync(d_u, uniforms, nB * (nK + 1) * 4, cudaMemcpyHostToDevice, s) ==
                   cudaSuccess;
    if (!ok) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    rc = launch(ctx, d_logits, logits_dtype, K > 0 ? d_q : nullptr, K > 0 ? d_tok : nullptr, d_u,
                B, K, V, temperature, d_len, d_out, K > 0 ? d_mask : nullptr,
                row_stats ? d_stats : nullptr, p_draft ? d_pd : nullptr, status ? d_st : nullptr,
                s);
    if (rc != SV_OK)
        return rc;
    ok = cudaMemcpyAsync(accept_len, d_len, nB * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaMemcpyAsync(out_tokens, d_out, nB * (nK + 1) * 4, cudaMemcpyDeviceToHost, s) ==
             cudaSuccess;
    if (K > 0)
        ok = ok && cudaMemcpyAsync(accept_mask, d_mask, nB * nK, cudaMemcpyDeviceToHost, s) ==
                       cudaSuccess;
    if (row_stats)
        ok = ok && cudaMemcpyAsync(row_stats, d_stats, nB * (nK + 1) * 8, cudaMemcpyDeviceToHost,
                                   s) == cudaSuccess;
    if (p_draft && K > 0)
        ok = ok && cudaMemcpyAsync(p_draft, d_pd, nB * nK * 4, cudaMemcpyDeviceToHost, s) ==
                       cudaSuccess;
    if (status)
        ok = ok && cudaMemcpyAsync(status, d_st, nB * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    if (!ok) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return spec_verify_get_error(ctx, stream, nullptr);
}

}  // extern "C"
