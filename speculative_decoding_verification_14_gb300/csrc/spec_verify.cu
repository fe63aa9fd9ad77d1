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
// Design (one launch per call; no global workspace besides a 4-byte error word):
//  * one thread-block cluster of C CTAs per sequence; CTA r owns a contiguous
//    vocabulary slice of every row, and each warp of the CTA owns a contiguous
//    stretch of that slice;
//  * every warp streams its stretch through a private ring of shared-memory
//    stages filled by cp.async.bulk (the TMA bulk-copy engine), each stage
//    completing on its own mbarrier -- warps never wait for one another inside
//    a row, and shared memory does not grow with the vocabulary;
//  * lanes keep a running (max, sum of exponentials) with packed f32x2
//    arithmetic; each warp publishes one partial per row;
//  * each warp pushes its 16-byte partial into a slot of every CTA of the
//    cluster with st.async, completing on that CTA's exchange mbarrier (armed
//    for the C x warps partials of the row), so no cluster barrier sits on
//    the per-row path; the first warp of a CTA to find a row's partials
//    complete merges them in a fixed order (double-float accumulation,
//    accurate exp2), takes the accept/reject decision and posts it in shared
//    memory for the CTA's other warps;
//  * rows are consumed in order and the loop stops at the first rejection,
//    like the pages' loop; a warp streams the next row while the decision on
//    the previous one is taken, and a rejection ends that stream;
//  * the residual (or bonus) draw streams the rejected draft row through the
//    same rings, records per-tile totals, meets the other CTAs' totals in
//    distributed shared memory, and one warp of the owning CTA locates the
//    token by warp-parallel scans;
//  * with the drafter's logits in place of q (the DL form), each test row's
//    draft row streams through the ring right after it, once the decision on
//    the previous row is settled, and yields a second partial per warp; the
//    test and the residual draw form q from the draft row's merged offset
//    and normaliser.
#include <cuda_runtime.h>
#include <cooperative_groups.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace {

using sv::kMaxK;
using sv::kMaxRows;
using sv::kChunkBytes;

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxWarps = 16;
constexpr int kChunkVecs = kChunkBytes / 16;  // 16-byte vectors per ring stage
constexpr int kVecPerLane = kChunkVecs / 32;
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
    uint32_t* al_hist;      // optional: one count per accepted length (0 = sequence error)
    const int32_t* offsets; // ragged batch: [B+1] packed row offsets (NULL: K rows for all)
    int64_t total_rows;     // ragged batch: rows in the packed arrays
    int64_t V;
    int64_t slice;          // vocabulary entries per CTA (multiple of 8)
    int B, K, C, G;
    int wvec;               // 16-byte vectors per warp stretch
    int ntw;                // draw tiles per warp stretch (capacity of the tile-total table)
    int off_fixed, off_bar, off_part, off_tt;  // shared-memory layout
    int bulk;               // 1: rows move with cp.async.bulk (16-byte aligned rows)
    int qvec;               // 1: draft rows move with cp.async.bulk as well
    int speculate;          // 1: first chunks of the next row are issued before the decision
    float c_hi, c_lo;       // log2(e)/T = c_hi + c_lo with c_lo > 0 (accurate paths)
    float c;                // log2(e)/T rounded to float (per-entry paths)
    float T;
    // draft logits in place of q (the DL kernels): q_i = softmax(d_i / T_d)
    const void* dlogits;    // [B, K, V] in the target's dtype
    float cd_hi, cd_lo;     // log2(e)/T_d split as c_hi, c_lo
    float cd;               // log2(e)/T_d rounded to float
};

struct FF {  // hi + lo, see the double-float helpers below
    float hi, lo;
};

// Fixed shared state of one CTA.  samp is written by every CTA of the cluster
// (st.async pushes), like the row partials.
struct __align__(16) SvShared {
    float4 samp[2][sv::kMaxCluster];  // pushed by every CTA: (total hi, total lo, bad, 0) per draw round
    FF wtot[kMaxWarps];
    int wbad[kMaxWarps];
    int x[kMaxK];
    float u[kMaxRows];
    float rs_m[kMaxRows];
    float rs_s[kMaxRows];
    float pd[kMaxK];
    // one-row steps: the warp that first finds a row's partials complete
    // decides it and posts the outcome here for the CTA's other warps
    int claim;     // rows claimed so far (row i is claimed by moving it from i to i + 1)
    int rec_row;   // the row whose outcome the record holds
    int rec_state, rec_code, rec_j, rec_mode, rec_ndec;
    float rec_A, rec_Shi, rec_Slo;
    float rec_Ad, rec_Sd;   // draft logits: the draft row's offset and normaliser
    float4 grp[kMaxRows];   // a group's row outcomes (amax, M, num, kind)
    float2 grpS[kMaxRows];  // ... and their normalisers (hi, lo)
    float2 grpD[kMaxRows];  // draft logits: the draft rows' (offset, normaliser)
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

// L2 eviction policy "evict first": for data read once (the draft row of a
// draw), so that it does not push out logits that a draw may read again.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// The bulk copy above with an L2 eviction policy.
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                                   unsigned long long* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
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

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// 16 bytes into another CTA's shared memory, counted as complete_tx on that
// CTA's mbarrier (the receiver waits on its own barrier, nobody else waits).
__device__ __forceinline__ void st_async_v4(uint32_t dst, float4 v, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(dst),
        "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
        "r"(__float_as_uint(v.w)), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Arrive with no memory ordering: used where the barrier only bounds CTA
// lifetimes and carries no data.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool mbar_test(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ int ld_acquire_cta(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_cta(int* p, int v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Slow path of a bounded wait: poll phase `parity` of `bar` until it
// completes or `limit_ns` passes (also after a fixed number of polls).  Between
// polls the warp sleeps with exponential backoff (32 ns up to 256 ns), so a
// waiting warp takes no issue slots from the warps that compute.  Returns
// false on give-up.
__device__ __noinline__ bool mbar_wait_slow(unsigned long long* bar, uint32_t parity,
                                            unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    unsigned sleep = 32;
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        __nanosleep(sleep);
        if (mbar_try_wait(bar, parity))
            return true;
        if (sleep < 256)
            sleep <<= 1;
        if ((it & 15u) == 15u && global_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

// Wait for phase `parity` of `bar`, giving up after `limit_ns`.  The first
// try_wait (which itself suspends the warp for a while) nearly always
// succeeds, so only that test is inline.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity))
        return true;
    return mbar_wait_slow(bar, parity, limit_ns);
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

// 2^y for y = hi + lo (y <= 8 here) to about one ulp, on the FMA pipe (used for the
// few values that must be accurate: merge weights and p(x)).  y = n + f with
// n = rint(hi) and |f| <= 1/2 (lo folded into f); 2^f = e^(f ln 2) by its
// Taylor series to degree 7 in (f ln 2), whose truncation error on that
// interval is below 1e-8 relative; 2^n is added to the exponent field (the
// result stays normal for n >= -125; below that the weight is 0, negligible
// next to the offset's own term of 1).
__device__ __forceinline__ float exp2_accurate(FF y) {
    if (!(y.hi > -125.f))
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
    return __int_as_float(__float_as_int(p) + ((int)n << 23));
}

// 2^((l - m) log2e/T) accurately; 0 for l = -inf.
__device__ __forceinline__ float exp2_diff_accurate(float l, float m, float c_hi, float c_lo) {
    if (!(l > -INFINITY))
        return 0.f;
    return exp2_accurate(exp2_arg_ff(l, m, c_hi, c_lo));
}

// ------------------------------------------------------------ elements -----
// Per-entry arithmetic.  An entry's weight is 2^y with y = (l - a) * c, where
// c = log2(e)/T rounded to float and `a` is a reference logit (an offset).
// Any offset gives the same softmax as long as every term of a sum, and the
// merge of the sums, agree on the offset each sum is taken against.  For bf16
// logits l - a is one mixed-precision subtraction (the bf16 operand is widened
// exactly inside the instruction), for fp32 logits one packed subtraction per
// pair; the product is one packed multiply per pair.

// l - a for the two bf16 entries of a 32-bit word (na = -a)
__device__ __forceinline__ float2 bf16x2_minus(uint32_t w, float na) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %3;\n\t"
        "add.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w), "f"(na));
    return make_float2(lo, hi);
}

template <int ES>
struct Elem;
template <>
struct Elem<4> {
    static constexpr int E = 4;  // entries per 16-byte vector
    static constexpr uint32_t kNegInf = 0xff800000u;
    using Max = float;  // running max of raw values (NaN-propagating)
    __device__ static __forceinline__ Max max_init() { return -INFINITY; }
    __device__ static __forceinline__ Max vmax(const uint4 w, Max m) {
        return fmax_nan(fmax_nan(m, fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y))),
                        fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    __device__ static __forceinline__ Max mmax(Max a, Max b) { return fmax_nan(a, b); }
    __device__ static __forceinline__ float value(Max m) { return m; }
    __device__ static __forceinline__ void diff(const uint4 w, float na, float2 (&d)[2]) {
        const float2 n2 = make_float2(na, na);
        d[0] = __fadd2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), n2);
        d[1] = __fadd2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), n2);
    }
    __device__ static __forceinline__ float load(const void* base, int64_t idx) {
        return __ldg(static_cast<const float*>(base) + idx);
    }
    __device__ static __forceinline__ uint32_t load_raw(const void* base, int64_t idx) {
        return __ldg(static_cast<const uint32_t*>(base) + idx);
    }
};
template <>
struct Elem<2> {
    static constexpr int E = 8;
    static constexpr uint32_t kNegInf = 0xff80u;
    using Max = uint32_t;  // running max of raw values as bf16x2 (NaN-propagating)
    __device__ static __forceinline__ Max max_init() { return 0xff80ff80u; }
    __device__ static __forceinline__ Max vmax(const uint4 w, Max m) {
        return bf16x2_max_nan(m, bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w)));
    }
    __device__ static __forceinline__ Max mmax(Max a, Max b) { return bf16x2_max_nan(a, b); }
    __device__ static __forceinline__ float value(Max m) { return fmax_nan(bf16_lo(m), bf16_hi(m)); }
    __device__ static __forceinline__ void diff(const uint4 w, float na, float2 (&d)[4]) {
        d[0] = bf16x2_minus(w.x, na);
        d[1] = bf16x2_minus(w.y, na);
        d[2] = bf16x2_minus(w.z, na);
        d[3] = bf16x2_minus(w.w, na);
    }
    __device__ static __forceinline__ float load(const void* base, int64_t idx) {
        const unsigned short h = __ldg(static_cast<const unsigned short*>(base) + idx);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ static __forceinline__ uint32_t load_raw(const void* base, int64_t idx) {
        return __ldg(static_cast<const unsigned short*>(base) + idx);
    }
};

// ------------------------------------------------------- warp helpers -----

// Floats as ints in the same order (any NaN above +inf), so that one integer
// warp reduction gives the float maximum.
__device__ __forceinline__ int ord_key(float f) {
    const int i = f != f ? 0x7fffffff : __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord_val(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// NaN-propagating maximum over the warp, in every lane
__device__ __forceinline__ float warp_max_nan(float v) {
    return ord_val(__reduce_max_sync(kFull, ord_key(v)));
}

// Sums over the warp, reduced in one fixed order and broadcast from lane 0 so
// that every lane (and every warp doing the same reduction) holds the same bits.
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

// Inclusive double-float scan over the first n lanes (lanes >= n hold
// whatever arrives; callers ignore them).  log2(n) steps instead of five.
__device__ __forceinline__ FF warp_incl_scan_n(FF v, int n) {
    const int lane = threadIdx.x & 31;
    for (int o = 1; o < n; o <<= 1) {
        const FF u = shfl_up_ff(v, o);
        if (lane >= o)
            v = ff_add(v, u);
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
// Only lanes below `n` take part.  Returns -1 only if every part is 0.
__device__ __forceinline__ int pick_lane(float part, FF incl, FF rem, int n, int& take_last) {
    const int lane = threadIdx.x & 31;
    const unsigned cross = __ballot_sync(kFull, lane < n && !take_last && ff_gt(incl, rem));
    if (cross)
        return __ffs(cross) - 1;
    const unsigned pos = __ballot_sync(kFull, lane < n && part > 0.f);
    take_last = 1;
    return pos ? 31 - __clz(pos) : -1;
}

// One 16-byte vector of a row stretch from global memory with element loads,
// entries at or past `lim` reading as -inf (rows that are not 16-byte aligned).
template <int ES>
__device__ __forceinline__ uint4 load_vec_elems(const void* logits, int64_t gbase, int64_t e,
                                                int64_t lim) {
    constexpr int E = Elem<ES>::E;
    uint32_t r[E];
#pragma unroll
    for (int k = 0; k < E; ++k)
        r[k] = e + k < lim ? Elem<ES>::load_raw(logits, gbase + e + k) : Elem<ES>::kNegInf;
    if constexpr (ES == 4)
        return make_uint4(r[0], r[1], r[2], r[3]);
    else
        return make_uint4(r[0] | (r[1] << 16), r[2] | (r[3] << 16), r[4] | (r[5] << 16),
                          r[6] | (r[7] << 16));
}

// ------------------------------------------------------- row statistics -----

// Sum over this lane's vectors of one chunk (vector k*32 + lane of `buf`, for
// k*32 + lane < nv) of 2^((l - a) c), with TRACK folding the raw values into
// the NaN-propagating max `mx` on the way.  Returned as two parts: with SPLIT
// the sums over the chunk's two halves (vectors k < kVecPerLane / 2, and the
// rest: a bf16 chunk's two draw tiles), without it the sum and 0, taken in
// two packed accumulators alternating within a vector (shorter dependency
// chains; the draft-logit form measured faster with them).
template <int ES, bool FULL, bool TRACK, bool SPLIT = true>
__device__ __forceinline__ float2 fold_chunk(const uint4* buf, int nv, float a, float c,
                                             typename Elem<ES>::Max& mx) {
    constexpr int E = Elem<ES>::E;
    const int lane = threadIdx.x & 31;
    const float2 c2 = make_float2(c, c);
    const float na = -a;
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
        if (FULL || k * 32 + lane < nv) {
            const uint4 w = buf[k * 32 + lane];
            if constexpr (TRACK)
                mx = Elem<ES>::vmax(w, mx);
            float2 d[E / 2];
            Elem<ES>::diff(w, na, d);
#pragma unroll
            for (int h = 0; h < E / 2; ++h) {
                const float2 y = __fmul2_rn(d[h], c2);
                const float2 e = make_float2(ex2_approx(y.x), ex2_approx(y.y));
                if (SPLIT ? k < kVecPerLane / 2 : !(h & 1))
                    s0 = __fadd2_rn(s0, e);
                else
                    s1 = __fadd2_rn(s1, e);
            }
        }
    }
    if constexpr (!SPLIT) {
        const float2 t = __fadd2_rn(s0, s1);
        return make_float2(t.x + t.y, 0.f);
    }
    return make_float2(s0.x + s0.y, s1.x + s1.y);
}

// One lane's running partial of a row: offset a, sum s of 2^((l - a) c) over
// the entries seen so far, NaN-propagating max mx of the raw values.
//
// The offset starts at the max of the lane's entries in the row's first chunk
// and moves only when a later chunk holds an entry more than 8 binades above
// it (or a NaN / inf): the offset then moves up to that chunk's max, the sum
// so far is rescaled and the chunk is summed again.  Accepted terms are
// therefore at most 2^8 (no overflow, and y's rounding stays small for the
// terms that dominate), and the offset is always the value of an entry the
// lane has seen, so its own term keeps s >= 1 and terms that underflow are
// negligible.  The per-chunk max pass of a textbook online softmax is gone.
// With `track` the max is kept exactly (the reported row statistics are taken
// against the row max); without it a chunk is accepted on its sum alone: a
// sum of at most kFoldBound = (entries per lane per chunk) x 2^8 means every
// term is at most kFoldBound, and a larger (or NaN / inf) sum sends the chunk
// through the max and the rules above.  SPLIT: see fold_chunk.
template <int ES, bool SPLIT = true>
struct LaneSum {
    static constexpr float kFoldBound = (float)(kVecPerLane * Elem<ES>::E * 256);
    float a, s;
    typename Elem<ES>::Max mx;

    __device__ __forceinline__ void start(const uint4* buf, int nv) {
        const int lane = threadIdx.x & 31;
        s = 0.f;
        mx = Elem<ES>::max_init();
        typename Elem<ES>::Max m0 = Elem<ES>::max_init();
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k)
            if (k * 32 + lane < nv)
                m0 = Elem<ES>::vmax(buf[k * 32 + lane], m0);
        a = Elem<ES>::value(m0);
    }

    // Folds one chunk in; returns the lane's sums over the chunk's two halves
    // (vectors k < kVecPerLane / 2 and the rest) against the offset `a` holds
    // afterwards (zero when the chunk adds nothing).
    __device__ __forceinline__ float2 chunk(const uint4* buf, int nv, float c, bool track) {
        typename Elem<ES>::Max cm = Elem<ES>::max_init();
        float2 hs;
        float cs, m;
        if (track) {
            hs = nv == kChunkVecs ? fold_chunk<ES, true, true, SPLIT>(buf, nv, a, c, cm)
                                  : fold_chunk<ES, false, true, SPLIT>(buf, nv, a, c, cm);
            cs = hs.x + hs.y;
            mx = Elem<ES>::mmax(mx, cm);
            m = Elem<ES>::value(cm);
        } else {
            hs = nv == kChunkVecs ? fold_chunk<ES, true, false, SPLIT>(buf, nv, a, c, cm)
                                  : fold_chunk<ES, false, false, SPLIT>(buf, nv, a, c, cm);
            cs = hs.x + hs.y;
            if (cs <= kFoldBound) {  // false for NaN
                s += cs;
                return hs;
            }
            const int lane = threadIdx.x & 31;
#pragma unroll
            for (int k = 0; k < kVecPerLane; ++k)
                if (k * 32 + lane < nv)
                    cm = Elem<ES>::vmax(buf[k * 32 + lane], cm);
            m = Elem<ES>::value(cm);
        }
        if ((m - a) * c <= 8.f) {  // false for NaN, +inf, or no offset yet
            s += cs;
            return hs;
        }
        if (!(m < INFINITY)) {  // NaN or +inf: the row is poisoned through mx; stop summing
            a = INFINITY;
            s = 0.f;
            return make_float2(0.f, 0.f);
        }
        if (!(m > -INFINITY))  // an all -inf chunk seen with no offset yet adds nothing
            return make_float2(0.f, 0.f);
        s = s > 0.f ? s * ex2_approx((a - m) * c) : 0.f;
        a = m;
        typename Elem<ES>::Max unused = Elem<ES>::max_init();
        hs = fold_chunk<ES, false, false, SPLIT>(buf, nv, a, c, unused);
        s += hs.x + hs.y;
        return hs;
    }
};

// ----------------------------------------------------------------- draw -----

// Draw weights of the E entries of one vector against the row offset a and
// normaliser S (double-float in the caller, its high part here):
//   RESID: S * max(0, p - q) = max(0, 2^((l - a) c) - q S)  (residual draw)
//   else : S * p             = 2^((l - a) c)                (bonus / target row)
// Entries at or past n weigh 0.  With RESID the bit patterns of q fold into
// qbits (unsigned max) for the range check.  Returns the sum of the weights.
template <int ES, bool RESID, bool MASK = true>
__device__ __forceinline__ float entry_weights(const uint4 lv, const float (&qq)[Elem<ES>::E], int n,
                                               float na, float c, float S,
                                               float (&w)[Elem<ES>::E], uint32_t& qbits) {
    constexpr int E = Elem<ES>::E;
    const float2 c2 = make_float2(c, c), nS = make_float2(-S, -S);
    float2 d[E / 2];
    Elem<ES>::diff(lv, na, d);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < E / 2; ++h) {
        const float2 y = __fmul2_rn(d[h], c2);
        float2 e = make_float2(ex2_approx(y.x), ex2_approx(y.y));
        if constexpr (RESID) {
            e = __ffma2_rn(make_float2(qq[2 * h], qq[2 * h + 1]), nS, e);
            e.x = fmaxf(e.x, 0.f);
            e.y = fmaxf(e.y, 0.f);
            qbits = __vimax3_u32(qbits, __float_as_uint(qq[2 * h]), __float_as_uint(qq[2 * h + 1]));
        }
        if (MASK && n < E) {
            if (2 * h >= n)
                e.x = 0.f;
            if (2 * h + 1 >= n)
                e.y = 0.f;
        }
        w[2 * h] = e.x;
        w[2 * h + 1] = e.y;
        acc = __fadd2_rn(acc, e);
    }
    return acc.x + acc.y;
}

// Draft logits: the E entries of one vector of draft row j as q_v S_d scaled
// to the target side, 2^((d_v - a_d) c_d) (nad = -a_d); the caller multiplies
// by S / S_d.  The pass and the locate step of the residual draw both call
// this, so both see the same weights.
template <int ES>
__device__ __forceinline__ void draft_q(const uint4 dv, float nad, float cd, float (&qq)[Elem<ES>::E]) {
    constexpr int E = Elem<ES>::E;
    float2 d[E / 2];
    Elem<ES>::diff(dv, nad, d);
    const float2 c2 = make_float2(cd, cd);
#pragma unroll
    for (int h = 0; h < E / 2; ++h) {
        const float2 y = __fmul2_rn(d[h], c2);
        qq[2 * h] = ex2_approx(y.x);
        qq[2 * h + 1] = ex2_approx(y.y);
    }
}

// q values of a residual draw are valid when each is in [0, +inf) (-0 counts
// as 0): as unsigned bit patterns, below the +inf pattern, or exactly -0.
__device__ __forceinline__ bool q_bits_valid(uint32_t qbits) {
    return qbits < 0x7f800000u || qbits == 0x80000000u;
}

// --------------------------------------------------------------- kernel -----

// Residency target: sv::kThreadsPerSM threads per SM, seven CTAs of 128 (shared
// memory allows no more), so a thread may use up to 72 registers.
// DL: the drafter's logits in place of q.  Every test row's draft row then
// streams right after its target row through the same ring (q_i needs the draft
// row's own maximum and normaliser), each warp publishes a second partial for
// it, the test is u * q(x) < p(x) with q(x) = 2^((d_x - a_d) c_d) / S_d, and
// the residual draw reads the draft row's logits where it would read q.
template <int ES, int NT, int NS, bool DL>
__global__ void __launch_bounds__(NT, NS == sv::kStages ? sv::kThreadsPerSM / NT : sv::kDeepCtasPerSM)
    sv_verify_kernel(const __grid_constant__ SvArgs a) {
    constexpr int kStages = NS;  // ring stages per warp
    constexpr int E = Elem<ES>::E;
    constexpr int NW = NT / 32;
    static_assert(NW <= kMaxWarps, "too many warps");
    constexpr int kPer = (sv::kMaxCluster * NW + 31) / 32;  // merge partials per lane, at most
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)a.C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Sequence b's rows: b*(K+1) .. for a uniform batch; for a ragged one the
    // packed rows offsets[b] .. offsets[b+1]-1 (its own depth K_b), draft rows
    // from offsets[b] - b.  Offsets that describe no packing leave K = 0 and
    // nothing of the sequence is read or written but accept_len and status.
    int k_seq = a.K;
    int64_t r_seq = (int64_t)b * (a.K + 1), d_seq = (int64_t)b * a.K;
    bool bad_off = false;
    if (a.offsets) {
        const int o0 = __ldg(a.offsets + b), o1 = __ldg(a.offsets + b + 1);
        bad_off = !(o0 >= b && o1 > o0 && o1 - o0 - 1 <= a.K &&
                    (int64_t)o1 + (a.B - 1 - b) <= a.total_rows);
        k_seq = bad_off ? 0 : o1 - o0 - 1;
        r_seq = bad_off ? 0 : o0;
        d_seq = bad_off ? 0 : (int64_t)o0 - b;
    }
    const int K = k_seq;
    const int64_t row0 = r_seq;   // first target row of sequence b
    const int64_t drow0 = d_seq;  // first draft row (and token, mask, p_draft entry)
    const int64_t V = a.V;
    const int C = a.C;
    const int G = a.G;
    const int GG = DL ? 2 * G : G;  // partial rows per parity: a draft partial per target row (DL)
    const float c = a.c;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    SvShared& sh = *reinterpret_cast<SvShared*>(smem_raw + a.off_fixed);
    unsigned long long* bar = reinterpret_cast<unsigned long long*>(smem_raw + a.off_bar);
    unsigned long long* xbar = bar + NW * kStages;  // [0..1] row partials by parity, [2..3] draw rounds
    float4* part = reinterpret_cast<float4*>(smem_raw + a.off_part);  // [2][GG][C*NW] (a, S.hi, S.lo, max)
    float* tt = reinterpret_cast<float*>(smem_raw + a.off_tt);          // [2][NW][ntw] draw tile totals, offsets
    unsigned char* ring = smem_raw + (size_t)warp * kStages * kChunkBytes;
    unsigned long long* wbar = bar + warp * kStages;

    // this CTA's slice and this warp's stretch of it (in 16-byte vectors)
    const int64_t v0 = (int64_t)rank * a.slice;
    const int64_t L = v0 < V ? (V - v0 < a.slice ? V - v0 : a.slice) : 0;
    const int nvec = (int)((L + E - 1) / E);
    const int wv0 = min(nvec, warp * a.wvec);
    const int wv1 = min(nvec, wv0 + a.wvec);
    const int wn = wv1 - wv0;
    const int nch = (wn + kChunkVecs - 1) / kChunkVecs;  // ring chunks per row

    if (lane == 0) {
        for (int st = 0; st < kStages; ++st)
            mbar_init(&wbar[st], 1);
        if (warp == 0)
            for (int k = 0; k < sv::kExchangeBarriers; ++k)
                mbar_init(&xbar[k], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (tid < K)
        sh.x[tid] = a.tokens[drow0 + tid];
    if (tid <= K)
        sh.u[tid] = a.u[row0 + tid];
    if (tid == 0) {
        sh.claim = 0;
        sh.rec_row = -1;
    }
    __syncthreads();
    // the exchange barriers must be initialised everywhere before the first
    // push: arrive now, wait just before pushing
    cluster_arrive();
    bool cluster_ready = false, cluster_left = false;

    // ---- per-warp stream through the private ring ----
    // stage indices and the consumer's phase bit advance incrementally; the
    // counters below are the same in every lane of the warp
    //
    // A copy into the warp's own stage depends on no other CTA and always
    // lands, so its wait has a long fixed limit of its own (sv::kCopyWaitNs,
    // five times the limit on waits for other CTAs); nothing at run time
    // shortens it.
    uint32_t st_issue = 0, st_wait = 0, ph_wait = 0;
    int in_flight = 0;
    bool timed_out = false;
    auto issue = [&](const void* src, uint32_t bytes, bool read_once = false) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&wbar[st_issue], bytes);
            if (read_once)
                bulk_copy_g2s_hint(ring + st_issue * kChunkBytes, src, bytes, &wbar[st_issue],
                                   l2_policy_evict_first());
            else
                bulk_copy_g2s(ring + st_issue * kChunkBytes, src, bytes, &wbar[st_issue]);
        }
        st_issue = st_issue == kStages - 1 ? 0 : st_issue + 1;
        ++in_flight;
    };
    auto wait_next = [&]() -> const uint4* {
        if (!mbar_wait_bounded(&wbar[st_wait], ph_wait, sv::kCopyWaitNs))
            timed_out = true;
        return reinterpret_cast<const uint4*>(ring + st_wait * kChunkBytes);
    };
    auto release = [&]() {
        __syncwarp();
        if (st_wait == kStages - 1) {
            st_wait = 0;
            ph_wait ^= 1u;
        } else {
            ++st_wait;
        }
        --in_flight;
    };
    const unsigned char* lstretch =
        static_cast<const unsigned char*>(a.logits) + (row0 * V + v0) * ES + (size_t)wv0 * 16;
    const size_t row_bytes = (size_t)V * ES;
    auto row_chunk_src = [&](int row, int ch) {
        return lstretch + (size_t)row * row_bytes + (size_t)ch * kChunkBytes;
    };
    auto row_chunk_bytes = [&](int ch) {
        return (uint32_t)(min(kChunkVecs, wn - ch * kChunkVecs) * 16);
    };
    // DL: this warp's stretch of draft row 0 (draft rows share the target's geometry)
    const unsigned char* dstretch =
        DL ? static_cast<const unsigned char*>(a.dlogits) + (drow0 * V + v0) * ES + (size_t)wv0 * 16
           : nullptr;

    // The row stream: (iss_row, iss_ch) is the next chunk to issue.  Chunks go
    // out up to kStages ahead of consumption, across row boundaries, but never
    // past row lim_row.  DL: a test row's draft row (iss_half 1) follows it.
    int iss_row = 0, iss_ch = 0, iss_half = 0, lim_row = (G < K + 1 ? G : K + 1) - 1;
    const unsigned char* iss_src = lstretch;
    const uint32_t last_bytes = nch > 0 ? row_chunk_bytes(nch - 1) : 0u;
    auto top_up = [&]() {
        if (nch == 0)
            return;
        while (in_flight < kStages && iss_row <= lim_row) {
            issue(iss_src, iss_ch == nch - 1 ? last_bytes : (uint32_t)kChunkBytes);
            if (++iss_ch == nch) {
                iss_ch = 0;
                if (DL && iss_half == 0 && iss_row < K) {
                    iss_half = 1;
                    iss_src = dstretch + (size_t)iss_row * row_bytes;
                } else {
                    iss_half = 0;
                    ++iss_row;
                    iss_src = row_chunk_src(iss_row, 0);
                }
            } else {
                iss_src += kChunkBytes;
            }
        }
    };
    // the first chunks of row 0 go out before the inputs are checked
    if (a.bulk && !bad_off)
        top_up();

    // ---- validation (every warp takes the same decision) ----
    int state = kStateRun, code = SV_OK;
    {
        const bool bad_x = __any_sync(kFull, lane < K && (sh.x[lane] < 0 || (int64_t)sh.x[lane] >= V));
        const float ul = lane <= K ? sh.u[lane] : 0.5f;
        const float uh = (lane == 0 && K == kMaxK) ? sh.u[kMaxK] : 0.5f;
        const bool bad_u = __any_sync(kFull, !(ul >= 0.f && ul < 1.f) || !(uh >= 0.f && uh < 1.f));
        if (bad_off) {
            state = kStateError;
            code = SV_ERR_BAD_OFFSETS;
        } else if (bad_x) {
            state = kStateError;
            code = SV_ERR_TOKEN_RANGE;
        } else if (bad_u) {
            state = kStateError;
            code = SV_ERR_UNIFORM_RANGE;
        }
    }
    // lane i: l(x_i), and q(x_i) -- or, from draft logits, d_x_i -- in every warp
    float lx_lane = 0.f, qx_lane = 0.f;
    if (state == kStateRun && lane < K) {
        const int x = sh.x[lane];
        lx_lane = Elem<ES>::load(a.logits, (row0 + lane) * V + x);
        qx_lane = DL ? Elem<ES>::load(a.dlogits, (drow0 + lane) * V + x)
                     : __ldg(a.q + (drow0 + lane) * V + x);
    }
    const int P = C * NW;  // row partials per row: every warp of the cluster
    const bool track = a.row_stats != nullptr;  // the row max is reported
    uint32_t xph = 0;      // phase bits of the two row-partial barriers

    // ---- the test loop: rows in order ([P1]) ----
    int j = -1, ndec = 0, mode = kModeBonus;
    float rowA = 0.f;
    FF rowS = {0.f, 0.f};
    float rowAd = 0.f, rowSd = 1.f;  // DL: the rejected row's draft offset and normaliser

    // Streams this warp's stretch of row `row` into ls.  After every chunk
    // poll() may end the stream (returns false): a decision arrived that
    // makes the row unnecessary.
    // The bonus row K also leaves, per draw tile of this warp's stretch, the
    // warp's sum of 2^((l - a_w) c) and the offset a_w it is taken against
    // (the lanes' largest offset when the tile's chunk was folded), so a
    // bonus draw needs no second pass over the row.  (Not in the draft-logit
    // form, which sums its chunks unsplit and keeps the pass.)
    constexpr int kTilesPerChunk = kChunkVecs * E / sv::kDrawTile;  // 2 (bf16) or 1 (f32)
    static_assert(kTilesPerChunk == 1 || kTilesPerChunk == 2, "draw tiles per chunk");
    float* const tt_w = tt + warp * a.ntw;          // this warp's tile totals
    float* const tta_w = tt + (NW + warp) * a.ntw;  // ... and their offsets
    auto record_tiles = [&](int ch, float2 hs, float la, float cc) {
        const float aw = warp_max_nan(la);
        const float sc = (aw > -INFINITY && aw < INFINITY) ? ex2_approx((la - aw) * cc) : 0.f;
        const float t0 = warp_sum_bcast((kTilesPerChunk == 2 ? hs.x : hs.x + hs.y) * sc);
        const float t1 = kTilesPerChunk == 2 ? warp_sum_bcast(hs.y * sc) : 0.f;
        const int t = ch * kTilesPerChunk;
        if (lane == 0) {
            tt_w[t] = t0;
            tta_w[t] = aw;
            if (kTilesPerChunk == 2 && t + 1 < a.ntw) {
                tt_w[t + 1] = t1;
                tta_w[t + 1] = aw;
            }
        }
    };

    // (DL: half 1 streams the draft row of `row` at c_d, without the exact max)
    auto stream_row = [&](int row, LaneSum<ES, !DL>& ls, auto&& poll, int half = 0) -> bool {
        const float cc = half ? a.cd : c;
        const bool trk = half ? false : track;
        const bool tiles = !DL && row == K && half == 0;
        ls.a = -INFINITY;
        ls.s = 0.f;
        ls.mx = Elem<ES>::max_init();
        for (int ch = 0; ch < nch; ++ch) {
            const int nv = min(kChunkVecs, wn - ch * kChunkVecs);
            const uint4* buf;
            if (a.bulk) {
                top_up();
                buf = wait_next();
            } else {
                // rows that are not 16-byte aligned: element loads into the
                // warp's current stage, then the same arithmetic
                uint4* dst = reinterpret_cast<uint4*>(ring + st_wait * kChunkBytes);
                const int64_t gbase = (half ? drow0 : row0) * V + (int64_t)row * V + v0;
                const void* src = half ? a.dlogits : a.logits;
                const int64_t cv = (int64_t)wv0 + (int64_t)ch * kChunkVecs;
                for (int k = 0; k < kVecPerLane; ++k)
                    if (k * 32 + lane < nv)
                        dst[k * 32 + lane] = load_vec_elems<ES>(src, gbase, (cv + k * 32 + lane) * E, L);
                __syncwarp();
                buf = dst;
            }
            if (ch == 0)
                ls.start(buf, nv);
            const float2 hs = ls.chunk(buf, nv, cc, trk);
            if (tiles)
                record_tiles(ch, hs, ls.a, cc);
            if (a.bulk)
                release();
            else
                __syncwarp();
            if (!poll())
                return false;
        }
        return true;
    };

    // This warp's partial of a row -- offset = the lanes' largest, sum in
    // double-float, NaN-propagating max -- pushed into slot (par, r) of every
    // CTA of the cluster.
    // (DL: half 1 publishes the draft row's partial, at c_d, into slot r + G)
    auto publish = [&](int par, int r, const LaneSum<ES, !DL>& ls, int half = 0) {
        const float aw = warp_max_nan(ls.a);
        const float mw = (track && !half) ? warp_max_nan(Elem<ES>::value(ls.mx)) : aw;
        FF sw = {0.f, 0.f};
        const float2 ch = half ? make_float2(a.cd_hi, a.cd_lo) : make_float2(a.c_hi, a.c_lo);
        if (ls.s > 0.f && aw < INFINITY)
            sw = two_prod(ls.s, exp2_diff_accurate(ls.a, aw, ch.x, ch.y));
        const FF Sw = warp_sum_bcast(sw);
        const bool any_to = __any_sync(kFull, timed_out);
        if (!cluster_ready) {
            cluster_wait();
            cluster_ready = true;
        }
        if (lane < C) {
            const uint32_t slot = smem_addr(&part[(par * GG + r + (half ? G : 0)) * P + rank * NW + warp]);
            st_async_v4(mapa_shared(slot, lane), make_float4(aw, any_to ? -1.f : Sw.hi, Sw.lo, mw),
                        mapa_shared(smem_addr(&xbar[par]), lane));
        }
    };

    // Waits (bounded) for the partials of slot `par`.
    auto wait_partials = [&](int par) {
        // (exchange waits outlast a peer's own bounded ring waits, so a late
        // peer's push lands before anyone gives up on it)
        if (!mbar_wait_bounded(&xbar[par], (xph >> par) & 1u, 3 * sv::kWaitNs))
            timed_out = true;
        xph ^= 1u << par;
    };

    // The combined statistics of row i and what its test concluded.
    struct RowOutcome {
        float amax, M, num;
        FF S;
        int kind;  // 0 accept, 1 reject (or bonus row), 2 timeout, 3 non-finite
        float ad;  // DL: the draft row's offset ...
        FF Sd;     // ... and normaliser
    };
    // The C * NW partials in slot (par, r): their largest offset, NaN-
    // propagating max and sum against that offset, merged in a fixed order
    // (c2 = (c_hi, c_lo) of the row's temperature).  Sets `to` when a warp
    // timed out.
    auto merge_slot = [&](int slot, bool xto, float2 c2, float& amax, float& M, bool& to) -> FF {
        float4 pv[kPer];
        float mloc = -INFINITY;
        amax = -INFINITY;
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
            const int p = lane + 32 * t;
            pv[t] = make_float4(-INFINITY, 0.f, 0.f, -INFINITY);
            if (p < P && !xto) {
                pv[t] = part[slot * P + p];
                amax = fmaxf(amax, pv[t].x);
                mloc = fmax_nan(mloc, pv[t].w);
                to |= pv[t].y < 0.f;
            }
        }
        M = warp_max_nan(mloc);
        amax = ord_val(__reduce_max_sync(kFull, ord_key(amax)));  // (offsets are never NaN)
        // (a NaN or inf entry poisons its lane's offset to +inf, an all -inf
        // row leaves every offset at -inf: both show in the merged offset)
        FF acc = {0.f, 0.f};
        if (amax > -INFINITY && amax < INFINITY) {
#pragma unroll
            for (int t = 0; t < kPer; ++t)
                if (pv[t].y > 0.f) {
                    const float wgt = exp2_diff_accurate(pv[t].x, amax, c2.x, c2.y);
                    FF term = two_prod(pv[t].y, wgt);
                    term.lo = fmaf(pv[t].z, wgt, term.lo);
                    acc = ff_add(acc, term);
                }
        }
        return warp_sum_bcast(acc);
    };
    // A warp combines the partials of row i (slot par, r) and evaluates
    // [P1]'s test for it.
    auto merge_row = [&](int i, int par, int r) -> RowOutcome {
        const bool xto = __any_sync(kFull, timed_out);
        bool to = false;
        RowOutcome o;
        o.ad = 0.f;
        o.Sd = FF{0.f, 0.f};
        // (DL: the draft row's slot too, through the same code)
        for (int h = 0; h < ((DL && i < K) ? 2 : 1); ++h) {
            float am, mm;
            const FF Sx = merge_slot(par * GG + r + (h ? G : 0), xto,
                                     h ? make_float2(a.cd_hi, a.cd_lo) : make_float2(a.c_hi, a.c_lo),
                                     am, mm, to);
            if (h == 0) {
                o.S = Sx;
                o.amax = am;
                o.M = mm;
            } else {
                o.Sd = Sx;
                o.ad = am;
            }
        }
        const bool finite = o.amax > -INFINITY && o.amax < INFINITY;
        const bool dfinite = !(DL && i < K) || (o.ad > -INFINITY && o.ad < INFINITY);
        const float lxi = __shfl_sync(kFull, lx_lane, i & 31);
        const float qxf = __shfl_sync(kFull, qx_lane, i & 31);  // DL: d(x_i)
        // lane 1: 2^((l_x - a) c); DL, lane 2: 2^((d_x - a_d) c_d)
        float num = 0.f;
        const bool dl2 = DL && lane == 2;
        if ((lane == 1 || dl2) && (dl2 ? dfinite : finite) && i < K)
            num = exp2_diff_accurate(dl2 ? qxf : lxi, dl2 ? o.ad : o.amax, dl2 ? a.cd_hi : a.c_hi,
                                     dl2 ? a.cd_lo : a.c_lo);
        const float numd = DL ? __shfl_sync(kFull, num, 2) : 0.f;
        o.num = __shfl_sync(kFull, num, 1);
        if (xto || __any_sync(kFull, to))
            o.kind = 2;
        else if (!finite || !dfinite || (!DL && i < K && !(qxf >= 0.f && qxf < INFINITY)))
            o.kind = 3;
        else if (i == K)
            o.kind = 1;
        else if (DL)  // u < p(x)/q(x) as u * 2^((d_x - a_d) c_d) * S < 2^((l_x - a) c) * S_d
            o.kind = ff_gt(ff_mul(FF{o.num, 0.f}, o.Sd), ff_mul(two_prod(sh.u[i], numd), o.S)) ? 0 : 1;
        else  // u < p(x)/q(x) as u * q(x) * S < 2^((l_x - a) c)
            o.kind = ff_gt(FF{o.num, 0.f}, ff_mul(two_prod(sh.u[i], qxf), o.S)) ? 0 : 1;
        return o;
    };
    // The loop of [P1] acting on row i's outcome; `writer` warps also record
    // the optional per-row outputs.
    auto apply_row = [&](int i, const RowOutcome& o, bool writer) {
        if (o.kind == 2) {
            state = kStateError;
            code = SV_ERR_TIMEOUT;
            return;
        }
        if (o.kind == 3 && !(o.amax > -INFINITY && o.amax < INFINITY)) {
            state = kStateError;
            code = SV_ERR_NONFINITE;
            return;
        }
        if (writer && lane == 0 && a.row_stats) {
            // reported against the row max: S * 2^((a - M) c)
            sh.rs_m[i] = __fdiv_rn(o.M, a.T);
            const float w = exp2_diff_accurate(o.amax, o.M, a.c_hi, a.c_lo);
            sh.rs_s[i] = fmaf(o.S.lo, w, o.S.hi * w);
        }
        ndec = i + 1;
        if (o.kind == 3) {  // the draft probability of x_i is not a probability
            state = kStateError;
            code = SV_ERR_NONFINITE;
            return;
        }
        if (i < K && writer && lane == 0 && a.p_draft)
            sh.pd[i] = __fdiv_rn(o.num, o.S.hi);
        if (o.kind == 1) {
            state = kStateSample;
            j = i;
            mode = i < K ? kModeResidual : kModeBonus;
            rowA = o.amax;
            rowS = o.S;
            if (DL && i < K) {
                rowAd = o.ad;
                rowSd = o.Sd.hi;
            }
        }
    };
    auto decide = [&](int i, int par, int r) { apply_row(i, merge_row(i, par, r), true); };

    if (G == 1) {
        // Rows stream back to back: while row cur streams, the partials of row
        // cur - 1 arrive, and the decision on it is taken between two chunks.
        // A rejection there ends the stream, so the next row is read only as
        // far as it got before the decision (a few chunks per warp).
        int cur = 0, pend = -1;
        // One warp per CTA decides a row -- the first to find its partials
        // complete -- and posts the outcome; the others pick it up.
        auto take_record = [&]() {
            state = sh.rec_state;
            code = sh.rec_code;
            j = sh.rec_j;
            mode = sh.rec_mode;
            ndec = sh.rec_ndec;
            rowA = sh.rec_A;
            rowS = FF{sh.rec_Shi, sh.rec_Slo};
            if (DL) {
                rowAd = sh.rec_Ad;
                rowSd = sh.rec_Sd;
            }
        };
        auto record_posted = [&](int i) {
            // every lane acquires, so each lane's reads of the record follow it
            return __all_sync(kFull, ld_acquire_cta(&sh.rec_row) >= i);
        };
        auto decide_claimed = [&](int i) -> bool {  // true if this warp decided row i
            int won = 0;
            if (lane == 0)
                won = atomicCAS(&sh.claim, i, i + 1) == i;
            if (!__shfl_sync(kFull, won, 0))
                return false;
            decide(i, i & 1, 0);
            if (lane == 0) {
                sh.rec_state = state;
                sh.rec_code = code;
                sh.rec_j = j;
                sh.rec_mode = mode;
                sh.rec_ndec = ndec;
                sh.rec_A = rowA;
                sh.rec_Shi = rowS.hi;
                sh.rec_Slo = rowS.lo;
                if (DL) {
                    sh.rec_Ad = rowAd;
                    sh.rec_Sd = rowSd;
                }
                st_release_cta(&sh.rec_row, i);
            }
            __syncwarp();
            return true;
        };
        // non-blocking: the decision on row `pend` if it can be had now
        auto poll = [&]() -> bool {
            if (pend < 0)
                return true;
            const int pp = pend & 1;
            if (record_posted(pend)) {
                take_record();
            } else {
                const bool ready = __shfl_sync(kFull, (int)mbar_test(&xbar[pp], (xph >> pp) & 1u), 0) != 0;
                if (!ready || !decide_claimed(pend))
                    return true;
            }
            xph ^= 1u << pp;
            pend = -1;
            return state == kStateRun;
        };
        // blocking (bounded): the decision on row i
        auto settle_row = [&](int i) {
            const int pp = i & 1;
            if (!record_posted(i)) {
                wait_partials(pp);  // flips xph
                if (!decide_claimed(i)) {
                    const unsigned long long t0 = global_ns();
                    while (!record_posted(i)) {
                        __nanosleep(64);
                        if (global_ns() - t0 > 4 * sv::kWaitNs) {
                            state = kStateError;
                            code = SV_ERR_TIMEOUT;
                            return;
                        }
                    }
                    take_record();
                }
                return;
            }
            take_record();
            xph ^= 1u << pp;
        };
        while (state == kStateRun) {
            const int pc = cur & 1;
            if (tid == 0)
                mbar_arrive_expect_tx(&xbar[pc], (uint32_t)(P * 16 * ((DL && cur < K) ? 2 : 1)));
            lim_row = cur < K ? cur + 1 : K;
            // (DL: the draft row streams after the decision on the previous
            // row is settled, so of a row the loop does not reach no more
            // than the ring's lookahead into its draft row is read)
            bool stopped = false;
            for (int h = 0; h < ((DL && cur < K) ? 2 : 1); ++h) {
                LaneSum<ES, !DL> ls;
                if (!stream_row(cur, ls, poll, h)) {
                    stopped = true;
                    break;
                }
                if (pend >= 0) {  // the decision on the previous row is still open
                    settle_row(pend);
                    pend = -1;
                    if (state != kStateRun) {
                        stopped = true;
                        break;
                    }
                }
                publish(pc, 0, ls, h);
            }
            if (stopped)
                break;
            pend = cur;
            if (cur == K) {  // the bonus row: nothing left to stream
                settle_row(cur);
                pend = -1;
                break;
            }
            ++cur;
        }
    } else {
        // Groups of G rows: every row of a group streams, the partials of the
        // whole group meet, and the rows are decided in order.
        int par = 0, g0 = 0;
        auto no_poll = []() { return true; };
        while (state == kStateRun) {
            const int ng = G < K + 1 - g0 ? G : K + 1 - g0;
            const int nd = DL ? max(0, min(ng, K - g0)) : 0;  // rows with a draft row
            if (tid == 0)
                mbar_arrive_expect_tx(&xbar[par], (uint32_t)(P * (ng + nd) * 16));
            lim_row = g0 + ng - 1;
            for (int r = 0; r < ng; ++r)
                for (int h = 0; h < (r < nd ? 2 : 1); ++h) {
                    LaneSum<ES, !DL> ls;
                    (void)stream_row(g0 + r, ls, no_poll, h);
                    publish(par, r, ls, h);
                }
            // the first chunks of the next group go out before the decision
            const int g1 = g0 + ng;
            if (a.bulk && a.speculate && g1 <= K) {
                lim_row = min(K, g1 + G - 1);
                top_up();
            }
            wait_partials(par);
            // the group's rows are combined in parallel, one warp per row,
            // then every warp walks the outcomes in order
            for (int r = warp; r < ng; r += NW) {
                const RowOutcome o = merge_row(g0 + r, par, r);
                if (lane == 0) {
                    sh.grp[r] = make_float4(o.amax, o.M, o.num, __int_as_float(o.kind));
                    sh.grpS[r] = make_float2(o.S.hi, o.S.lo);
                    if (DL)
                        sh.grpD[r] = make_float2(o.ad, o.Sd.hi);
                }
            }
            __syncthreads();
            for (int r = 0; r < ng && state == kStateRun; ++r) {
                const float4 g4 = sh.grp[r];
                const float2 g2 = sh.grpS[r];
                RowOutcome o;
                o.amax = g4.x;
                o.M = g4.y;
                o.num = g4.z;
                o.kind = __float_as_int(g4.w);
                o.S = FF{g2.x, g2.y};
                if (DL) {
                    const float2 gd = sh.grpD[r];
                    o.ad = gd.x;
                    o.Sd = FF{gd.y, 0.f};
                }
                apply_row(g0 + r, o, warp == 0);
            }
            __syncthreads();  // the outcome slots are reused by the next group
            par ^= 1;
            g0 = g1;
        }
    }
    // speculative chunks that will not be used: let them land before the ring is reused
    while (in_flight > 0) {
        (void)wait_next();
        release();
    }

    // ---- corrected or bonus draw over row j ([P1]) ----
    // This warp's stretch of row j is walked in tiles of kDrawTile entries: a
    // tile's draft probabilities are one ring stage, and lane l takes vectors
    // k*32 + l (k < kDV) of the tile's logits, loaded one tile ahead (an L2
    // prefetch of the whole stretch measured slower: in a full batch it only
    // adds to the DRAM queues).  Every tile's weight total goes to `tt` for
    // the locate step.
    constexpr int kDrawTile = sv::kDrawTile;    // entries per draw tile
    constexpr int kDV = kDrawTile / (32 * E);   // logits vectors per lane per tile
    const int64_t e0 = (int64_t)wv0 * E;
    const int64_t nq = max((int64_t)0, min((int64_t)wv1 * E, L) - e0);  // entries in this stretch
    const int nq32 = (int)nq;
    const int ntile = (nq32 + kDrawTile - 1) / kDrawTile;
    const unsigned char* lrow = nullptr;
    const float* qrow = nullptr;
    const unsigned char* drow = nullptr;  // DL: draft row j's slice
    int owner = -1, take_last = 0;
    FF rem = {0.f, 0.f};
    // the residual's q scale: S, or with draft logits S / S_d (see draft_q)
    const float Sf = (DL && j < K) ? __fdiv_rn(rowS.hi, rowSd) : rowS.hi;
    const int64_t gbase_j = (row0 + j) * V + v0;    // element index of the slice start
    const int64_t dgbase_j = (drow0 + j) * V + v0;  // DL: the same in the draft logits
    if (state == kStateSample) {
        lrow = static_cast<const unsigned char*>(a.logits) + ((row0 + j) * V + v0) * ES;
        if (DL)
            drow = j < K ? static_cast<const unsigned char*>(a.dlogits) + dgbase_j * ES : nullptr;
        else
            qrow = j < K ? a.q + (drow0 + j) * V + v0 : nullptr;
        const float na = -rowA;
        int sp = 0;
        const unsigned char* lbase = lrow + e0 * ES;
        const float* qbase = qrow ? qrow + e0 : nullptr;
        const unsigned char* dbase = drow ? drow + e0 * ES : nullptr;
        uint32_t qbits = 0;
        auto load_logits = [&](int t, uint4 (&lv)[kDV]) {
#pragma unroll
            for (int k = 0; k < kDV; ++k) {
                const int ve = t * kDrawTile + (k * 32 + lane) * E;
                if (ve >= nq32)
                    lv[k] = make_uint4(0, 0, 0, 0);
                else if (a.bulk)
                    lv[k] = __ldg(reinterpret_cast<const uint4*>(lbase + (size_t)ve * ES));
                else
                    lv[k] = load_vec_elems<ES>(a.logits, gbase_j + e0, ve, nq32);
            }
        };
        auto pass = [&](auto resid_tag) -> FF {
            constexpr bool RESID = decltype(resid_tag)::value;
            const bool use_ring = RESID && a.qvec;
            FF wacc = {0.f, 0.f};
            int qissued = 0;
            // the draft row's stages go out up to kStages tiles ahead -- one
            // for a rejection in the first half of the drafts: such a draw
            // has the most time before the batch's last sequences finish,
            // and its copies in flight would lengthen the memory queues the
            // rows of the sequences still testing wait in
            auto q_top_up = [&](int t) {
                while (qissued < ntile && qissued < t + (2 * j < K ? 1 : kStages)) {
                    if (DL)
                        issue(dbase + (size_t)qissued * kDrawTile * ES,
                              (uint32_t)(min(kDrawTile, nq32 - qissued * kDrawTile) * ES), true);
                    else
                        issue(qbase + (size_t)qissued * kDrawTile,
                              (uint32_t)(min(kDrawTile, nq32 - qissued * kDrawTile) * 4), true);
                    ++qissued;
                }
            };
            if (use_ring)
                q_top_up(0);
            auto tile_done = [&](int t, float ts) {
                const float tot = warp_sum_bcast(ts);
                if (lane == 0)
                    tt_w[t] = tot;
                wacc = ff_add(wacc, tot);
            };
            // Full tiles of 16-byte aligned rows: no masks, a pointer that
            // advances a tile at a time, the next tile's logits in flight.
            const int nfull = (a.bulk && (use_ring || !RESID)) ? nq32 / kDrawTile : 0;
            if (nfull > 0) {
                const float2 c2 = make_float2(c, c), nS = make_float2(-Sf, -Sf);
                const uint4* lp = reinterpret_cast<const uint4*>(lbase) + lane;
                uint4 lv[kDV];
#pragma unroll
                for (int k = 0; k < kDV; ++k)
                    lv[k] = __ldg(lp + k * 32);
                for (int t = 0; t < nfull; ++t) {
                    uint4 cur[kDV];
#pragma unroll
                    for (int k = 0; k < kDV; ++k)
                        cur[k] = lv[k];
                    if (t + 1 < nfull) {
                        lp += kDrawTile * ES / 16;
#pragma unroll
                        for (int k = 0; k < kDV; ++k)
                            lv[k] = __ldg(lp + k * 32);
                    }
                    const float4* q4 = nullptr;
                    if constexpr (RESID)
                        q4 = reinterpret_cast<const float4*>(wait_next());
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < kDV; ++k) {
                        float2 d[E / 2];
                        Elem<ES>::diff(cur[k], na, d);
                        float2 qp[E / 2];
                        if constexpr (RESID && DL) {
                            float qd[E];
                            draft_q<ES>(reinterpret_cast<const uint4*>(q4)[k * 32 + lane], -rowAd, a.cd, qd);
#pragma unroll
                            for (int h = 0; h < E / 2; ++h)
                                qp[h] = make_float2(qd[2 * h], qd[2 * h + 1]);
                        } else if constexpr (RESID) {
#pragma unroll
                            for (int h = 0; h < E / 4; ++h) {
                                const float4 v4 = q4[(k * 32 + lane) * (E / 4) + h];
                                qp[2 * h] = make_float2(v4.x, v4.y);
                                qp[2 * h + 1] = make_float2(v4.z, v4.w);
                            }
                        }
#pragma unroll
                        for (int h = 0; h < E / 2; ++h) {
                            const float2 y = __fmul2_rn(d[h], c2);
                            float2 e = make_float2(ex2_approx(y.x), ex2_approx(y.y));
                            if constexpr (RESID) {
                                e = __ffma2_rn(qp[h], nS, e);
                                e.x = fmaxf(e.x, 0.f);
                                e.y = fmaxf(e.y, 0.f);
                                if (!DL)
                                    qbits = __vimax3_u32(qbits, __float_as_uint(qp[h].x),
                                                         __float_as_uint(qp[h].y));
                            }
                            acc = __fadd2_rn(acc, e);
                        }
                    }
                    if (use_ring) {
                        release();
                        q_top_up(t + 1);
                    }
                    tile_done(t, acc.x + acc.y);
                }
            }
            // the rest: a partial last tile, or rows that need element loads
            for (int t = nfull; t < ntile; ++t) {
                uint4 lv[kDV];
                load_logits(t, lv);
                const float* qs = nullptr;
                if (use_ring) {
                    q_top_up(t);
                    qs = reinterpret_cast<const float*>(wait_next());
                }
                float ts = 0.f;
#pragma unroll
                for (int k = 0; k < kDV; ++k) {
                    const int vi = k * 32 + lane;  // vector within the tile
                    const int ve = t * kDrawTile + vi * E;
                    const int n = min(E, max(0, nq32 - ve));
                    float qq[E];
                    if constexpr (RESID && DL) {
                        // (entries at or past n weigh 0 whatever qq holds there)
                        const uint4 dv = use_ring ? reinterpret_cast<const uint4*>(qs)[vi]
                                                  : load_vec_elems<ES>(a.dlogits, dgbase_j + e0, ve, nq32);
                        draft_q<ES>(dv, -rowAd, a.cd, qq);
#pragma unroll
                        for (int h = 0; h < E; ++h)
                            if (h >= n)
                                qq[h] = 0.f;
                    } else if constexpr (RESID) {
                        if (use_ring) {
                            const float4* q4 = reinterpret_cast<const float4*>(qs + vi * E);
#pragma unroll
                            for (int h = 0; h < E / 4; ++h) {
                                const float4 v4 = 4 * h < n ? q4[h] : make_float4(0.f, 0.f, 0.f, 0.f);
                                qq[4 * h] = v4.x;
                                qq[4 * h + 1] = v4.y;
                                qq[4 * h + 2] = v4.z;
                                qq[4 * h + 3] = v4.w;
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < E; ++h)
                                qq[h] = h < n ? __ldg(qbase + ve + h) : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < E; ++h)
                            qq[h] = 0.f;
                    }
                    float w[E];
                    ts += entry_weights<ES, RESID, true>(lv[k], qq, n, na, c, Sf, w, qbits);
                }
                if (use_ring)
                    release();
                tile_done(t, ts);
            }
            return wacc;
        };
        // The bonus draw's tile totals from the row pass: each rescaled from
        // its offset to the row's merged offset, summed in tile order.
        auto bonus_from_tiles = [&]() -> FF {
            __syncwarp();  // lane 0's records are visible to the warp
            FF wacc = {0.f, 0.f};
            for (int t0 = 0; t0 < ntile; t0 += 32) {
                const int t = t0 + lane;
                float v = 0.f;
                if (t < ntile) {
                    const float tv = tt_w[t];
                    v = tv > 0.f ? tv * ex2_approx((tta_w[t] - rowA) * c) : 0.f;
                    tt_w[t] = v;
                }
                const int n = min(32, ntile - t0);
                for (int k = 0; k < n; ++k)
                    wacc = ff_add(wacc, __shfl_sync(kFull, v, k));
            }
            return wacc;
        };
        for (int round = 0; round < 2; ++round) {
            if (tid == 0)
                mbar_arrive_expect_tx(&xbar[2 + sp], (uint32_t)(C * 16));
            const FF wacc = mode == kModeResidual ? pass(std::true_type{})
                            : (!DL && mode == kModeBonus) ? bonus_from_tiles()
                                                  : pass(std::false_type{});
            const bool badq = __any_sync(kFull, !q_bits_valid(qbits));
            const bool to = __any_sync(kFull, timed_out);
            if (lane == 0) {
                sh.wtot[warp] = wacc;
                sh.wbad[warp] = to ? 2 : (badq ? 1 : 0);
            }
            __syncthreads();
            if (warp == 0) {
                FF tot = {0.f, 0.f};
                int bad = 0;
                for (int w2 = 0; w2 < NW; ++w2) {
                    tot = ff_add(tot, sh.wtot[w2]);
                    bad = max(bad, sh.wbad[w2]);
                }
                if (lane < C)
                    st_async_v4(mapa_shared(smem_addr(&sh.samp[sp][rank]), lane),
                                make_float4(tot.hi, tot.lo, (float)bad, 0.f),
                                mapa_shared(smem_addr(&xbar[2 + sp]), lane));
            }
            const bool dto = !mbar_wait_bounded(&xbar[2 + sp], 0u, 3 * sv::kWaitNs);
            FF ctot = {0.f, 0.f};
            int cbad = __any_sync(kFull, dto) ? 2 : 0;
            if (lane < C && !cbad) {
                const float4 v4 = sh.samp[sp][lane];
                ctot = FF{v4.x, v4.y};
                cbad = (int)v4.z;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1)
                cbad = max(cbad, __shfl_xor_sync(kFull, cbad, o));
            const FF incl = warp_incl_scan_n(ctot, C);
            const FF S = shfl_ff(incl, C - 1);
            const FF thr = ff_mul(FF{sh.u[K], 0.f}, S);
            take_last = 0;
            owner = pick_lane(ctot.hi, incl, thr, C, take_last);
            const FF excl = shfl_ff(warp_excl_from_incl(incl, FF{0.f, 0.f}), owner < 0 ? 0 : owner);
            if (cbad) {
                state = kStateError;
                code = cbad == 2 ? SV_ERR_TIMEOUT : SV_ERR_NONFINITE;
                break;
            }
            if (S.hi == 0.f && mode == kModeResidual) {
                // max(0, p - q) vanished (rounding or an unnormalised q):
                // draw from p_j itself with the same uniform
                mode = kModeTargetRow;
                sp ^= 1;
                continue;
            }
            if (owner < 0) {  // no positive weight anywhere: unreachable for a finite row max
                state = kStateError;
                code = SV_ERR_NONFINITE;
            }
            rem = ff_add(thr, ff_neg(excl));
            break;
        }
        // no CTA of the cluster touches another's shared memory after this
        // (every push into a CTA has landed before it passed the exchange)
        cluster_arrive_relaxed();
        cluster_left = true;

        if (state == kStateSample && rank == owner && warp == 0) {
            // Tile, then sub-tile, lane and entry.  The CTA's tiles in
            // vocabulary order are warp-major: flat index f = w * ntw + t, and
            // tiles past a warp's stretch weigh 0.  Lane l takes kTL
            // consecutive flat tiles per round, so one scan across lanes
            // covers 32 * kTL tiles.
            constexpr int kTL = 4;
            const int ntw = a.ntw;
            const int nflat = NW * ntw;
            auto tile_total = [&](int f) -> float {
                if (f >= nflat)
                    return 0.f;
                const int w = f / ntw, t = f - (f / ntw) * ntw;
                const int wv0w = min(nvec, w * a.wvec);
                const int nqw = (int)max((int64_t)0, min((int64_t)min(nvec, wv0w + a.wvec) * E, L) - (int64_t)wv0w * E);
                return t * kDrawTile < nqw ? tt[f] : 0.f;
            };
            int fsel = -1, flast = -1;
            FF carry = {0.f, 0.f}, at_sel = {0.f, 0.f}, at_last = {0.f, 0.f};
            for (int c0 = 0; c0 < nflat && fsel < 0; c0 += 32 * kTL) {
                float tv[kTL];
                FF ls_ = {0.f, 0.f};
#pragma unroll
                for (int k = 0; k < kTL; ++k) {
                    tv[k] = tile_total(c0 + lane * kTL + k);
                    ls_ = ff_add(ls_, tv[k]);
                }
                const FF in = ff_add(warp_incl_scan(ls_), carry);
                const FF ex = warp_excl_from_incl(in, carry);
                int tl = take_last;
                const int pk = pick_lane(ls_.hi, in, rem, 32, tl);
                if (pk >= 0) {
                    // within lane pk's kTL tiles, in order
                    FF run = shfl_ff(ex, pk);
                    int hit = -1, last = -1;
                    FF at_hit = {0.f, 0.f}, at_l = {0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < kTL; ++k) {
                        const float v = __shfl_sync(kFull, tv[k], pk);
                        const FF nxt = ff_add(run, v);
                        if (hit < 0 && !tl && ff_gt(nxt, rem)) {
                            hit = k;
                            at_hit = run;
                        }
                        if (v > 0.f) {
                            last = k;
                            at_l = run;
                        }
                        run = nxt;
                    }
                    if (hit >= 0) {
                        fsel = c0 + pk * kTL + hit;
                        at_sel = at_hit;
                    } else if (last >= 0) {
                        flast = c0 + pk * kTL + last;
                        at_last = at_l;
                    }
                }
                carry = shfl_ff(in, 31);
            }
            if (fsel < 0) {
                take_last = 1;
                fsel = max(flast, 0);
                at_sel = at_last;
            }
            rem = ff_add(rem, ff_neg(at_sel));
            const int ws = fsel / ntw, tsel = fsel - ws * ntw;
            const int wv0s = min(nvec, ws * a.wvec);
            const int64_t e0s = (int64_t)wv0s * E;
            const int nqs = (int)max((int64_t)0, min((int64_t)min(nvec, wv0s + a.wvec) * E, L) - e0s);
            // re-derive the tile's weights (the same arithmetic as the pass)
            float w[kDV][E], ts[kDV];
#pragma unroll
            for (int k = 0; k < kDV; ++k) {
                const int ve = tsel * kDrawTile + (k * 32 + lane) * E;
                const int n = min(E, max(0, nqs - ve));
                uint4 raw = make_uint4(0, 0, 0, 0);
                if (n > 0)
                    raw = a.bulk ? __ldg(reinterpret_cast<const uint4*>(lrow + (e0s + ve) * ES))
                                 : load_vec_elems<ES>(a.logits, gbase_j, e0s + ve, e0s + nqs);
                float qq[E];
                if (DL && mode == kModeResidual) {
                    uint4 dv = make_uint4(0, 0, 0, 0);
                    if (n > 0)
                        dv = a.qvec ? __ldg(reinterpret_cast<const uint4*>(drow + (e0s + ve) * ES))
                                    : load_vec_elems<ES>(a.dlogits, dgbase_j, e0s + ve, e0s + nqs);
                    draft_q<ES>(dv, -rowAd, a.cd, qq);
                } else if (mode == kModeResidual && a.qvec && n == E) {
#pragma unroll
                    for (int h = 0; h < E / 4; ++h) {
                        const float4 v4 = __ldg(reinterpret_cast<const float4*>(qrow + e0s + ve) + h);
                        qq[4 * h] = v4.x;
                        qq[4 * h + 1] = v4.y;
                        qq[4 * h + 2] = v4.z;
                        qq[4 * h + 3] = v4.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < E; ++h)
                        qq[h] = (mode == kModeResidual && h < n) ? __ldg(qrow + e0s + ve + h) : 0.f;
                }
                uint32_t qb = 0;
                ts[k] = mode == kModeResidual
                            ? entry_weights<ES, true>(raw, qq, n, -rowA, c, Sf, w[k], qb)
                            : entry_weights<ES, false>(raw, qq, n, -rowA, c, rowS.hi, w[k], qb);
            }
            // sub-tile k holds tile entries [k*32*E, (k+1)*32*E)
            int ksel = -1, klast = -1;
            FF run = {0.f, 0.f}, at_k = {0.f, 0.f}, at_klast = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kDV; ++k) {
                const float sk = warp_sum_bcast(ts[k]);
                const FF nxt = ff_add(run, sk);
                if (ksel < 0 && !take_last && ff_gt(nxt, rem)) {
                    ksel = k;
                    at_k = run;
                }
                if (sk > 0.f) {
                    klast = k;
                    at_klast = run;
                }
                run = nxt;
            }
            if (ksel < 0) {
                take_last = 1;
                ksel = max(klast, 0);
                at_k = at_klast;
            }
            rem = ff_add(rem, ff_neg(at_k));
            float tk = 0.f, wk[E];
#pragma unroll
            for (int k = 0; k < kDV; ++k)
                if (k == ksel) {
                    tk = ts[k];
#pragma unroll
                    for (int h = 0; h < E; ++h)
                        wk[h] = w[k][h];
                }
            const float inc = warp_incl_scan(tk);
            const int pk = pick_lane(tk, FF{inc, 0.f}, rem, 32, take_last);
            float prev = __shfl_up_sync(kFull, inc, 1);
            if (lane == 0)
                prev = 0.f;
            const int src = pk < 0 ? 0 : pk;
            const float ex = __shfl_sync(kFull, prev, src);
            // the entry: lane pk's E weights spread over lanes 0..E-1, one scan
            float we = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float v = __shfl_sync(kFull, wk[e], src);
                if (lane == e)
                    we = v;
            }
            const FF ine = ff_add(warp_incl_scan_n(FF{we, 0.f}, E), FF{ex, 0.f});
            int tle = take_last;
            int e = pick_lane(we, ine, rem, E, tle);
            if (e < 0)
                e = 0;
            const int tok = (int)(v0 + e0s + tsel * kDrawTile + (ksel * 32 + src) * E + e);
            // outputs of a finished sequence
            for (int i = lane; i <= K; i += 32) {
                a.out_tokens[row0 + i] = i < j ? sh.x[i] : (i == j ? tok : -1);
                if (i < K)
                    a.accept_mask[drow0 + i] = i < j ? 1 : 0;
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

    // ---- rank 0 reports the per-row statistics, or the sequence error ----
    if (rank == 0 && warp == 0) {
        const bool err = state == kStateError;
        const int nd = err ? 0 : ndec;
        for (int i = lane; i <= K && !bad_off; i += 32) {
            if (a.row_stats) {
                a.row_stats[(row0 + i) * 2] = i < nd ? sh.rs_m[i] : NAN;
                a.row_stats[(row0 + i) * 2 + 1] = i < nd ? sh.rs_s[i] : NAN;
            }
            if (i < K && a.p_draft)
                a.p_draft[drow0 + i] = i < nd ? sh.pd[i] : NAN;
            if (err) {
                a.out_tokens[row0 + i] = -1;
                if (i < K)
                    a.accept_mask[drow0 + i] = 0;
            }
        }
        if (err && lane == 0) {
            a.accept_len[b] = 0;
            if (a.status)
                a.status[b] = code;
            atomicOr(a.err_word, 1u << code);
            if (a.al_hist)
                atomicAdd(a.al_hist, 1u);
        }
    }

    // copies still in flight (only after an error) land before the exit
    while (in_flight > 0) {
        (void)wait_next();
        release();
    }
    // nobody leaves before every CTA is past its last push into the others
    if (!cluster_ready)
        cluster_wait();
    if (!cluster_left)
        cluster_arrive();
    cluster_wait();
}

// ----------------------------------------------------------------- host -----

using KernelFn = void (*)(SvArgs);

// dl: the draft-logit form (128 threads only)
KernelFn pick_kernel(int es, int threads, int stages = sv::kStages, bool dl = false) {
    constexpr int S3 = sv::kStages, S6 = sv::kStagesDeep;
    if (dl) {
        if (threads != 128 || (stages != S3 && stages != S6))
            return nullptr;
        if (es == 2)
            return stages == S6 ? sv_verify_kernel<2, 128, S6, true> : sv_verify_kernel<2, 128, S3, true>;
        return stages == S6 ? sv_verify_kernel<4, 128, S6, true> : sv_verify_kernel<4, 128, S3, true>;
    }
    if (stages == S6) {
        if (threads != 128)
            return nullptr;
        return es == 2 ? sv_verify_kernel<2, 128, S6, false> : sv_verify_kernel<4, 128, S6, false>;
    }
    if (es == 2) {
        if (threads == 128) return sv_verify_kernel<2, 128, S3, false>;
        if (threads == 256) return sv_verify_kernel<2, 256, S3, false>;
        if (threads == 512) return sv_verify_kernel<2, 512, S3, false>;
    } else {
        if (threads == 128) return sv_verify_kernel<4, 128, S3, false>;
        if (threads == 256) return sv_verify_kernel<4, 256, S3, false>;
        if (threads == 512) return sv_verify_kernel<4, 512, S3, false>;
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
    int greedy_max_cluster = 8;
    uint32_t* d_err = nullptr;
    int ovr_cluster = 0, ovr_group = 0, ovr_threads = 0;  // spec_verify_set_plan_override
    uint32_t* al_hist = nullptr;  // caller's accepted-length counters (device), or none
    int al_bins = 0;
    // staging for the host-buffer entry point
    unsigned char* d_stage = nullptr;
    size_t stage_bytes = 0;
};

namespace {

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
    return spec_verify_plan_for(ctx->num_sms, ctx->smem_optin, ctx->max_cluster, B, K, V, dtype,
                                ctx->ovr_cluster, ctx->ovr_group, ctx->ovr_threads, plan);
}

// (log2(e) / T) as hi + lo, hi just below the exact value so that lo is
// strictly positive: a -inf logit then gives -inf * lo = -inf, not NaN
void split_log2e_over(float T, float* hi, float* lo, float* rounded) {
    const double c_d = 1.4426950408889634074 / (double)T;
    *hi = (float)c_d;
    if ((double)*hi >= c_d)
        *hi = std::nextafter(*hi, 0.0f);
    *lo = (float)(c_d - (double)*hi);
    *rounded = (float)c_d;
}

// The draft-logit form's extra inputs (see spec_verify_run_draft_logits).
struct DraftLogits {
    const void* dlogits;  // [B, K, V], the target's dtype
    float T_draft;
};

int launch(sv_ctx* ctx, const void* logits, int dtype, const float* q, const int32_t* tokens,
           const float* uniforms, int B, int K, int64_t V, float T, int32_t* accept_len,
           int32_t* out_tokens, uint8_t* accept_mask, float* row_stats, float* p_draft,
           int32_t* status, cudaStream_t stream, const int32_t* offsets = nullptr,
           int64_t total_rows = 0, const DraftLogits* dl = nullptr) {
    if (ctx->al_hist && K + 2 > ctx->al_bins)
        return SV_ERR_INVALID_ARG;
    sv_plan plan;
    const int es = dtype == SV_BF16 ? 2 : 4;
    int rc = dl ? spec_verify_get_plan_draft_logits(ctx, B, K, V, dtype, 0, &plan)
                : make_plan(ctx, B, K, V, dtype, &plan);
    if (rc != SV_OK)
        return rc;
    KernelFn fn = pick_kernel(es, plan.threads, plan.stages, dl != nullptr);
    if (!fn)
        return SV_ERR_UNSUPPORTED;

    const sv::Layout lay = sv::layout_for(plan.slice, es, dl ? 2 * plan.group : plan.group,
                                          plan.threads, plan.cluster, plan.stages);
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
    args.al_hist = ctx->al_hist;
    args.offsets = offsets;
    args.total_rows = total_rows;
    args.V = V;
    args.slice = plan.slice;
    args.B = B;
    args.K = K;
    args.C = plan.cluster;
    args.G = plan.group;
    args.wvec = (int)lay.wvec;
    args.ntw = (int)lay.ntw;
    args.off_fixed = (int)lay.off_fixed;
    args.off_bar = (int)lay.off_bar;
    args.off_part = (int)lay.off_part;
    args.off_tt = (int)lay.off_tt;
    if (dl) {
        // target and draft rows share one chunk layout: the bulk copies only
        // when both are 16-byte aligned; qvec: draft row tiles through the ring
        args.q = nullptr;
        args.dlogits = K > 0 ? dl->dlogits : logits;  // K = 0: never read
        args.bulk = plan.bulk_copy && aligned(logits, 16) && aligned(args.dlogits, 16) ? 1 : 0;
        args.qvec = args.bulk;
        split_log2e_over(dl->T_draft, &args.cd_hi, &args.cd_lo, &args.cd);
    } else {
        args.bulk = plan.bulk_copy && aligned(logits, 16) ? 1 : 0;
        args.qvec = (V % 4 == 0) && q && aligned(q, 16) ? 1 : 0;
    }
    args.speculate = plan.prefetch_next && args.bulk ? 1 : 0;
    args.T = T;
    split_log2e_over(T, &args.c_hi, &args.c_lo, &args.c);

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

// What spec_verify_init and the no-allocation entry both need to know about a
// device before the first launch on it.
struct DeviceInfo {
    int num_sms = 0, smem_optin = 0;
    int max_cluster = 8;         // sampled verify kernel: largest usable cluster
    int greedy_max_cluster = 8;  // greedy kernel
};

// Device checks, kernel attributes and the largest usable clusters, with
// `device` current.  Shared by both entries so that their plans agree.
int device_setup(int device, DeviceInfo* info) {
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
    int max_cluster = 16;
    const int es_list[2] = {2, 4};
    // 0: the deep-ring kernel (128 threads); -1, -2: the draft-logit forms
    const int nt_list[6] = {128, 256, 512, 0, -1, -2};
    for (int es : es_list)
        for (int nt : nt_list) {
            KernelFn fn = nt > 0    ? pick_kernel(es, nt)
                          : nt == 0 ? pick_kernel(es, 128, sv::kStagesDeep)
                                    : pick_kernel(es, 128, nt == -1 ? sv::kStages : sv::kStagesDeep, true);
            if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin) != cudaSuccess) {
                (void)cudaGetLastError();
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
    info->num_sms = sms;
    info->smem_optin = optin;
    info->max_cluster = max_cluster;
    // the greedy kernel may use 16-CTA clusters only where the main kernel may
    info->greedy_max_cluster =
        (max_cluster >= 16 && sv::greedy_set_attributes() == 0) ? 16 : 8;
    return SV_OK;
}

void apply_device_info(sv_ctx* c, const DeviceInfo& info) {
    c->num_sms = info.num_sms;
    c->smem_optin = info.smem_optin;
    c->max_cluster = info.max_cluster;
    c->greedy_max_cluster = info.greedy_max_cluster;
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
        case SV_ERR_BAD_OFFSETS: return "ragged-batch row offsets describe no packing";
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
    DeviceInfo info;
    const int rc = device_setup(device, &info);
    if (rc != SV_OK)
        return rc;
    sv_ctx* ctx = new sv_ctx();
    ctx->device = device;
    ctx->max_B = max_B;
    ctx->max_K = max_K;
    ctx->max_V = max_V;
    apply_device_info(ctx, info);
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

int spec_verify_run_ragged(sv_ctx* ctx, const void* target_logits, int logits_dtype,
                           const float* q, const int32_t* draft_tokens, const float* uniforms,
                           const int32_t* row_offsets, int64_t total_rows, int B, int K_max,
                           int64_t V, float temperature, int32_t* accept_len,
                           int32_t* out_tokens, uint8_t* accept_mask, float* row_stats,
                           float* p_draft, int32_t* status, void* stream) {
    if (!ctx || !row_offsets || !aligned(row_offsets, 4))
        return SV_ERR_INVALID_ARG;
    if (B < 1 || K_max < 0 || total_rows < B || total_rows > (int64_t)B * (K_max + 1))
        return SV_ERR_INVALID_ARG;
    // the packed arrays are checked like a uniform batch of depth K_max; the
    // draft-side arrays are needed only if some sequence can have drafts
    const int rc = validate(ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B,
                            total_rows > B ? K_max : 0, V, temperature, accept_len, out_tokens,
                            accept_mask, row_stats, p_draft, status);
    if (rc != SV_OK)
        return rc;
    if ((double)total_rows * (double)V >= 1099511627776.0)  // 2^40
        return SV_ERR_INVALID_ARG;
    return launch(ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K_max, V,
                  temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft, status,
                  static_cast<cudaStream_t>(stream), row_offsets, total_rows);
}

int spec_verify_get_plan_truncated(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype,
                                   sv_plan* out) {
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    const int ovr = ctx->ovr_cluster > sv::kTruncMaxCluster ? sv::kTruncMaxCluster
                                                            : ctx->ovr_cluster;
    return spec_verify_plan_truncated_for(ctx->num_sms, ctx->max_cluster, B, K, V, logits_dtype,
                                          ovr, out);
}

int spec_verify_run_truncated(sv_ctx* ctx, const void* target_logits, int logits_dtype,
                              const float* q, const int32_t* draft_tokens, const float* uniforms,
                              int B, int K, int64_t V, float temperature, double top_p,
                              double min_p, int32_t* accept_len, int32_t* out_tokens,
                              uint8_t* accept_mask, float* row_stats, float* p_draft,
                              int32_t* status, void* stream) {
    const int rc = validate(ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K, V,
                            temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft,
                            status);
    if (rc != SV_OK)
        return rc;
    if (!(top_p > 0.0) || !(min_p < 1.0) || std::isnan(top_p) || std::isnan(min_p))
        return SV_ERR_INVALID_ARG;
    if (ctx->al_hist && K + 2 > ctx->al_bins)
        return SV_ERR_INVALID_ARG;
    sv_plan plan;
    const int prc = spec_verify_get_plan_truncated(ctx, B, K, V, logits_dtype, &plan);
    if (prc != SV_OK)
        return prc;
    const int es = logits_dtype == SV_BF16 ? 2 : 4;
    sv::TruncLaunch g;
    std::memset(&g, 0, sizeof g);
    g.logits = target_logits;
    g.q = q;
    g.tokens = draft_tokens;
    g.u = uniforms;
    g.accept_len = accept_len;
    g.out_tokens = out_tokens;
    g.accept_mask = accept_mask;
    g.row_stats = row_stats;
    g.p_draft = p_draft;
    g.status = status;
    g.err_word = ctx->d_err;
    g.al_hist = ctx->al_hist;
    g.V = V;
    g.slice = plan.slice;
    g.B = B;
    g.K = K;
    g.C = plan.cluster;
    g.es = es;
    g.vec = plan.bulk_copy && aligned(target_logits, 16) ? 1 : 0;
    g.qvec = (V % 4 == 0) && q && aligned(q, 16) ? 1 : 0;
    g.c = (float)(1.4426950408889634074 / (double)temperature);
    g.T = temperature;
    // min-p keeps l - l_max >= T ln(min_p); ln(min_p) = -inf for min_p <= 0 (off)
    g.dmin = min_p > 0.0 ? (float)((double)temperature * std::log(min_p)) : -INFINITY;
    g.top_p = top_p;
    g.wait_ns = sv::kWaitNs;
    DeviceGuard guard(ctx->device);
    return sv::trunc_launch(g, stream) == 0 ? SV_OK : SV_ERR_CUDA;
}

int spec_verify_get_plan_draft_logits(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype,
                                      int filters, sv_plan* out) {
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    const int cap = filters ? sv::kTruncMaxCluster : ctx->max_cluster;
    const int ovr = ctx->ovr_cluster > cap ? cap : ctx->ovr_cluster;
    return spec_verify_plan_draft_logits_for(ctx->num_sms, cap, B, K, V, logits_dtype, filters,
                                             ovr, out);
}

int spec_verify_run_draft_logits(sv_ctx* ctx, const void* target_logits, int logits_dtype,
                                 const void* draft_logits, const int32_t* draft_tokens,
                                 const float* uniforms, int B, int K, int64_t V,
                                 float temperature, float draft_temperature, double top_p,
                                 double min_p, int32_t* accept_len, int32_t* out_tokens,
                                 uint8_t* accept_mask, float* row_stats, float* p_draft,
                                 int32_t* status, void* stream) {
    const size_t es = logits_dtype == SV_BF16 ? 2 : 4;
    if (K > 0 && (!draft_logits || !aligned(draft_logits, es)))
        return SV_ERR_INVALID_ARG;
    // the shared checks want a float q for K > 0; the draft logits were
    // checked above, so a stand-in that passes those checks takes q's place
    static const float no_q = 0.f;
    const int rc = validate(ctx, target_logits, logits_dtype, K > 0 ? &no_q : nullptr,
                            draft_tokens, uniforms, B, K, V, temperature, accept_len, out_tokens,
                            accept_mask, row_stats, p_draft, status);
    if (rc != SV_OK)
        return rc;
    if (!(draft_temperature > 0.f) || !std::isfinite(draft_temperature))
        return SV_ERR_INVALID_ARG;
    if (!(top_p > 0.0) || !(min_p < 1.0) || std::isnan(top_p) || std::isnan(min_p))
        return SV_ERR_INVALID_ARG;
    if (ctx->al_hist && K + 2 > ctx->al_bins)
        return SV_ERR_INVALID_ARG;
    const int filters = (top_p < 1.0 || min_p > 0.0) ? 1 : 0;
    if (!filters) {
        // the plain verify with q formed from the draft logits: the main
        // kernel's draft-logit form
        const DraftLogits dl = {draft_logits, draft_temperature};
        return launch(ctx, target_logits, logits_dtype, nullptr, draft_tokens, uniforms, B, K, V,
                      temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft, status,
                      static_cast<cudaStream_t>(stream), nullptr, 0, &dl);
    }
    sv_plan plan;
    const int prc = spec_verify_get_plan_draft_logits(ctx, B, K, V, logits_dtype, filters, &plan);
    if (prc != SV_OK)
        return prc;
    sv::TruncLaunch g;
    std::memset(&g, 0, sizeof g);
    g.logits = target_logits;
    g.q = nullptr;
    g.dlogits = K > 0 ? draft_logits : target_logits;  // K = 0: never read
    g.tokens = draft_tokens;
    g.u = uniforms;
    g.accept_len = accept_len;
    g.out_tokens = out_tokens;
    g.accept_mask = accept_mask;
    g.row_stats = row_stats;
    g.p_draft = p_draft;
    g.status = status;
    g.err_word = ctx->d_err;
    g.al_hist = ctx->al_hist;
    g.V = V;
    g.slice = plan.slice;
    g.B = B;
    g.K = K;
    g.C = plan.cluster;
    g.es = (int)es;
    // target and draft rows share one unit layout: vectors only when both are aligned
    g.vec = plan.bulk_copy && aligned(target_logits, 16) && (K == 0 || aligned(draft_logits, 16))
                ? 1
                : 0;
    g.qvec = 0;
    g.c = (float)(1.4426950408889634074 / (double)temperature);
    g.cd = (float)(1.4426950408889634074 / (double)draft_temperature);
    g.T = temperature;
    g.dmin = min_p > 0.0 ? (float)((double)temperature * std::log(min_p)) : -INFINITY;
    g.top_p = top_p;
    g.wait_ns = sv::kWaitNs;
    DeviceGuard guard(ctx->device);
    return sv::trunc_launch(g, stream) == 0 ? SV_OK : SV_ERR_CUDA;
}

int spec_verify_get_plan_greedy(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype,
                                sv_plan* out) {
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    return spec_verify_plan_greedy_for(ctx->num_sms, ctx->greedy_max_cluster, B, K, V,
                                       logits_dtype, ctx->ovr_cluster, out);
}

int spec_verify_run_greedy(sv_ctx* ctx, const void* target_logits, int logits_dtype,
                           const int32_t* draft_tokens, int B, int K, int64_t V,
                           int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                           int32_t* row_argmax, int32_t* status, void* stream) {
    if (!ctx || !target_logits || !accept_len || !out_tokens)
        return SV_ERR_INVALID_ARG;
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16)
        return SV_ERR_INVALID_ARG;
    if (B < 1 || B > ctx->max_B || K < 0 || K > ctx->max_K || K > kMaxK || V < 1 ||
        V > ctx->max_V)
        return SV_ERR_INVALID_ARG;
    if ((double)B * (double)(K + 1) * (double)V >= 1099511627776.0)  // 2^40
        return SV_ERR_INVALID_ARG;
    if (K > 0 && (!draft_tokens || !accept_mask))
        return SV_ERR_INVALID_ARG;
    const int es = logits_dtype == SV_BF16 ? 2 : 4;
    if (!aligned(target_logits, es) || (draft_tokens && !aligned(draft_tokens, 4)) ||
        !aligned(accept_len, 4) || !aligned(out_tokens, 4) ||
        (row_argmax && !aligned(row_argmax, 4)) || (status && !aligned(status, 4)))
        return SV_ERR_INVALID_ARG;
    if (ctx->al_hist && K + 2 > ctx->al_bins)
        return SV_ERR_INVALID_ARG;
    sv_plan plan;
    const int rc = spec_verify_get_plan_greedy(ctx, B, K, V, logits_dtype, &plan);
    if (rc != SV_OK)
        return rc;
    sv::GreedyLaunch g;
    std::memset(&g, 0, sizeof g);
    g.logits = target_logits;
    g.tokens = draft_tokens;
    g.accept_len = accept_len;
    g.out_tokens = out_tokens;
    g.accept_mask = accept_mask;
    g.row_argmax = row_argmax;
    g.status = status;
    g.err_word = ctx->d_err;
    g.al_hist = ctx->al_hist;
    g.V = V;
    g.slice = plan.slice;
    g.B = B;
    g.K = K;
    g.C = plan.cluster;
    g.es = es;
    g.vec = plan.bulk_copy && aligned(target_logits, 16) ? 1 : 0;
    g.wait_ns = sv::kWaitNs;
    DeviceGuard guard(ctx->device);
    return sv::greedy_launch(g, stream) == 0 ? SV_OK : SV_ERR_CUDA;
}

int spec_verify_set_telemetry(sv_ctx* ctx, uint32_t* accept_hist, int bins) {
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    if (!accept_hist) {
        ctx->al_hist = nullptr;
        ctx->al_bins = 0;
        return SV_OK;
    }
    if (bins < 2 || !aligned(accept_hist, 4))
        return SV_ERR_INVALID_ARG;
    ctx->al_hist = accept_hist;
    ctx->al_bins = bins;
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

// ---------------------------------------------------------------------------
// spec_verify_run_noalloc: the verify of spec_verify_run without a context and
// without allocating anything.
//
// Who needs it: callers that cannot allocate device memory where they verify.
// A serving engine that reserved nearly all of HBM for its own pool (KV cache,
// activations) at start-up has nothing left for a library to cudaMalloc; a
// decode loop that must not pay the device-wide synchronisation cudaFree
// implies cannot own a context it later destroys; a plugin called through a
// fixed function table has no place to create or release one.
//
// What replaces the context: the kernel's only scratch is the word its
// sequence-error bits are ORed into.  Here that word is the first element of a
// file-scope device array (one copy per device, zero when the module is
// loaded), whose address is looked up once per device.  The device properties
// and kernel attributes that spec_verify_init queries are set up once per
// device, on the first call for it, in static host storage.
namespace {

constexpr int kNoAllocScratchWords = 64;  // 256 bytes of scratch per device
constexpr int kNoAllocScratchNeed = 1;    // words one call uses: the error word
constexpr int kNoAllocMaxDevices = 64;
constexpr int kNoAllocMaxB = 1 << 20;
constexpr int64_t kNoAllocMaxV = (int64_t)1 << 31;
static_assert(kNoAllocScratchNeed <= kNoAllocScratchWords, "scratch array too small");

static __device__ __align__(256) uint32_t sv_noalloc_scratch[kNoAllocScratchWords];

struct NoAllocDevice {
    std::atomic<int> ready{0};
    sv_ctx ctx;  // static storage: limits, planner inputs, scratch address
};
NoAllocDevice g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_setup_mutex;

// Everything spec_verify_init does except allocating: device checks, kernel
// attributes, the largest usable cluster, and the scratch address, all with
// `device` current.
int noalloc_setup(int device, sv_ctx* c) {
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    DeviceGuard guard(device);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != device) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    DeviceInfo info;
    const int rc = device_setup(device, &info);
    if (rc != SV_OK)
        return rc;
    uint32_t* scratch = nullptr;
    if (cudaGetSymbolAddress((void**)&scratch, sv_noalloc_scratch) != cudaSuccess || !scratch) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    c->device = device;
    c->max_B = kNoAllocMaxB;
    c->max_K = kMaxK;
    c->max_V = kNoAllocMaxV;
    apply_device_info(c, info);
    c->d_err = scratch;
    return SV_OK;
}

}  // namespace

extern "C" int spec_verify_run_noalloc(int device, const void* target_logits, int logits_dtype,
                                       const float* q, const int32_t* draft_tokens,
                                       const float* uniforms, int B, int K, int64_t V,
                                       float temperature, int32_t* accept_len,
                                       int32_t* out_tokens, uint8_t* accept_mask,
                                       float* row_stats, float* p_draft, int32_t* status,
                                       void* stream) {
    if (device < 0 || device >= kNoAllocMaxDevices)
        return SV_ERR_INVALID_ARG;
    NoAllocDevice& d = g_noalloc[device];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_noalloc_setup_mutex);
        if (!d.ready.load(std::memory_order_relaxed)) {
            const int rc = noalloc_setup(device, &d.ctx);
            if (rc != SV_OK)
                return rc;  // nothing cached: the next call tries again
            d.ready.store(1, std::memory_order_release);
        }
    }
    // sizes beyond this entry's limits (B <= 2^20, K <= 32, V <= 2^31) are
    // rejected here, before anything is launched
    const int rc = validate(&d.ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K,
                            V, temperature, accept_len, out_tokens, accept_mask, row_stats,
                            p_draft, status);
    if (rc != SV_OK)
        return rc;
    return launch(&d.ctx, target_logits, logits_dtype, q, draft_tokens, uniforms, B, K, V,
                  temperature, accept_len, out_tokens, accept_mask, row_stats, p_draft, status,
                  static_cast<cudaStream_t>(stream));
}
