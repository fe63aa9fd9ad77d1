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
//    bulk-copy engine) completing on an mbarrier, then two passes over shared
//    memory give the slice's max and sum of exponentials;
//  * the C partial (max, sum) pairs are combined through distributed shared
//    memory after a cluster barrier, in the same fixed order in every CTA, so
//    every CTA reaches the same accept/reject decision without broadcast;
//  * rows are consumed in order and the loop stops at the first rejection,
//    like the pages' loop, so rows after it are never read;
//  * the residual (or bonus) draw is split across the cluster too: each CTA
//    sums max(0, p - q) over its slice (q streamed from HBM, logits still in
//    shared memory), the per-CTA sums meet in distributed shared memory, and
//    only the CTA holding the crossing point re-scans one warp-sized stretch.
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
    int bulk;
    int qvec;
    float c_hi, c_lo;       // log2(e)/T split into two floats (hi + lo)
    double c_d;             // log2(e)/T in double
    double T_d;
    unsigned long long wait_ns;
};

// Fixed shared state of one CTA.  The part_* and samp_* members are read by
// the other CTAs of the cluster through distributed shared memory.
struct __align__(16) SvShared {
    unsigned long long mbar;
    float part_m[2][kMaxRows];
    float part_s[2][kMaxRows];
    int part_flag[2];
    double samp_tot[2];
    int samp_last[2];
    int samp_bad[2];
    int x[kMaxK];
    float u[kMaxRows];
    float lx[kMaxK];
    float qx[kMaxK];
    float rs_m[kMaxRows];
    float rs_s[kMaxRows];
    float pd[kMaxK];
    float red_f[32];
    int red_i[32];
    int state, j, code, ndec, mode, tok, owner;
    float rowM;
    double rowS;
    int loc_warp, loc_tile;
    double loc_rem;
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

// l - m for the exponent d*c_hi + d*c_lo.  A -inf logit (or -inf padding)
// would give d = -inf and, when c_lo < 0, -inf + inf = NaN; clamping d to a
// finite floor keeps the product with c_lo finite while d*c_hi still
// overflows to -inf, so the entry weighs exactly 0.  (NaN logits never reach
// this point: the row max propagates them and the row is rejected first.)
__device__ __forceinline__ float exp_arg_diff(float l, float m) { return fmaxf(l - m, -3.0e38f); }

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

// ------------------------------------------------------------ elements -----

template <int ES>
struct Elem;
template <>
struct Elem<4> {
    static constexpr int E = 4;  // entries per 16-byte vector
    static constexpr uint32_t kNegInf = 0xff800000u;
    __device__ static __forceinline__ void unpack(const uint4 w, float (&f)[4]) {
        f[0] = __uint_as_float(w.x);
        f[1] = __uint_as_float(w.y);
        f[2] = __uint_as_float(w.z);
        f[3] = __uint_as_float(w.w);
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
};
template <>
struct Elem<2> {
    static constexpr int E = 8;
    static constexpr uint32_t kNegInf = 0xff80u;
    __device__ static __forceinline__ void unpack(const uint4 w, float (&f)[8]) {
        f[0] = bf16_lo(w.x);
        f[1] = bf16_hi(w.x);
        f[2] = bf16_lo(w.y);
        f[3] = bf16_hi(w.y);
        f[4] = bf16_lo(w.z);
        f[5] = bf16_hi(w.z);
        f[6] = bf16_lo(w.w);
        f[7] = bf16_hi(w.w);
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

// ------------------------------------------------------- block helpers -----

template <int NT>
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Max over a staged row slice (nvec 16-byte vectors, padded with -inf).
// Every thread returns the same value.
template <int ES, int NT>
__device__ float slice_max(const unsigned char* buf, int nvec, SvShared& sh) {
    const int tid = threadIdx.x;
    float m;
    if constexpr (ES == 2) {
        uint32_t acc = 0xff80ff80u;
        for (int vi = tid; vi < nvec; vi += NT) {
            const uint4 w = reinterpret_cast<const uint4*>(buf)[vi];
            acc = bf16x2_max_nan(acc, w.x);
            acc = bf16x2_max_nan(acc, w.y);
            acc = bf16x2_max_nan(acc, w.z);
            acc = bf16x2_max_nan(acc, w.w);
        }
        m = fmax_nan(bf16_lo(acc), bf16_hi(acc));
    } else {
        m = -INFINITY;
        for (int vi = tid; vi < nvec; vi += NT) {
            const uint4 w = reinterpret_cast<const uint4*>(buf)[vi];
            m = fmax_nan(m, fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                                     fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w))));
        }
    }
    m = warp_max_nan<NT>(m);
    if ((tid & 31) == 0)
        sh.red_f[tid >> 5] = m;
    __syncthreads();
    float r = sh.red_f[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w)
        r = fmax_nan(r, sh.red_f[w]);
    __syncthreads();
    return r;
}

// sum_v 2^((l_v - m) * log2(e)/T) over a staged slice.  The exponent is formed
// as d*c_hi + d*c_lo with d = l - m exact for bf16 inputs, so the only
// rounding per entry is the final one and the ex2 approximation.
// Result valid in thread 0.
template <int ES, int NT>
__device__ float slice_sumexp(const unsigned char* buf, int nvec, float m, float c_hi, float c_lo,
                              SvShared& sh) {
    constexpr int E = Elem<ES>::E;
    const int tid = threadIdx.x;
    float s0 = 0.f, s1 = 0.f;
    for (int vi = tid; vi < nvec; vi += NT) {
        float f[E];
        Elem<ES>::unpack(reinterpret_cast<const uint4*>(buf)[vi], f);
#pragma unroll
        for (int k = 0; k < E; k += 2) {
            const float d0 = exp_arg_diff(f[k], m), d1 = exp_arg_diff(f[k + 1], m);
            s0 += ex2_approx(fmaf(d0, c_hi, d0 * c_lo));
            s1 += ex2_approx(fmaf(d1, c_hi, d1 * c_lo));
        }
    }
    float s = s0 + s1;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        s += __shfl_down_sync(kFull, s, o);
    if ((tid & 31) == 0)
        sh.red_f[tid >> 5] = s;
    __syncthreads();
    float r = 0.f;
    if (tid == 0)
        for (int w = 0; w < NT / 32; ++w)
            r += sh.red_f[w];
    __syncthreads();
    return r;
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

// Weights of one 16-byte vector of the staged row: residual max(0, p - q)
// (mode 0), unnormalised target weights exp(z - max) (modes 1 and 2).
// Entries at or past L weigh 0.  `bad` is raised by a NaN, infinite or
// negative q value.
template <int ES>
__device__ __forceinline__ void vec_weights(const unsigned char* buf, int vi, int64_t L,
                                            const float* qrow, int qvec, int mode, float M,
                                            float c_hi, float c_lo, float inv_s,
                                            float (&w)[Elem<ES>::E], bool& bad) {
    constexpr int E = Elem<ES>::E;
    float f[E];
    Elem<ES>::unpack(reinterpret_cast<const uint4*>(buf)[vi], f);
    const int64_t base = (int64_t)vi * E;
    float qq[E];
#pragma unroll
    for (int k = 0; k < E; ++k)
        qq[k] = 0.f;
    if (mode == kModeResidual) {
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
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const float d = exp_arg_diff(f[k], M);
        const float e = ex2_approx(fmaf(d, c_hi, d * c_lo));
        float wk;
        if (mode == kModeResidual) {
            const float qv = qq[k];
            if (base + k < L && !(qv >= 0.f && qv < INFINITY))
                bad = true;
            wk = fmaxf(e * inv_s - qv, 0.f);
        } else {
            wk = e;
        }
        w[k] = base + k < L ? wk : 0.f;
    }
}

// --------------------------------------------------------------- kernel -----

template <int ES, int NT>
__global__ void __launch_bounds__(NT) sv_verify_kernel(const __grid_constant__ SvArgs a) {
    constexpr int E = Elem<ES>::E;
    constexpr int NW = NT / 32;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)a.C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K;
    const int64_t V = a.V;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* bufs = smem_raw;
    SvShared& sh = *reinterpret_cast<SvShared*>(smem_raw + (size_t)a.G * a.rowbuf_bytes);
    float* wt = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(&sh) + sizeof(SvShared));

    // this CTA's vocabulary slice
    const int64_t v0 = (int64_t)rank * a.slice;
    const int64_t L = v0 < V ? (V - v0 < a.slice ? V - v0 : a.slice) : 0;
    const int nvec = (int)((L + E - 1) / E);
    const int64_t row0 = (int64_t)b * (K + 1);  // first logits row of this sequence

    if (tid == 0) {
        mbar_init(&sh.mbar, 1);
        fence_mbar_init();
        sh.part_flag[0] = sh.part_flag[1] = 0;
    }
    __syncthreads();

    uint32_t phase = 0;
    bool timed_out = false;

    // Moves rows g0 .. g0+ng-1 of this sequence's slice into shared memory.
    auto load_group = [&](int g0, int ng) {
        if (L == 0)
            return;
        if (a.bulk) {
            if (tid == 0) {
                fence_proxy_async();
                const uint32_t bytes = (uint32_t)(L * ES);
                mbar_arrive_expect_tx(&sh.mbar, bytes * (uint32_t)ng);
                for (int r = 0; r < ng; ++r) {
                    const unsigned char* src = static_cast<const unsigned char*>(a.logits) +
                                               ((row0 + g0 + r) * V + v0) * ES;
                    bulk_copy_g2s(bufs + (size_t)r * a.rowbuf_bytes, src, bytes, &sh.mbar);
                }
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
            const bool ok = mbar_wait_bounded(&sh.mbar, phase, a.wait_ns);
            phase ^= 1u;
            if (__syncthreads_or(!ok))
                timed_out = true;
        } else {
            __syncthreads();
        }
    };

    // first group's copy goes out before anything else
    const int G = a.G;
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
    // (made visible to thread 0 by the barriers below)

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
            const unsigned char* buf = bufs + (size_t)r * a.rowbuf_bytes;
            const float m = L ? slice_max<ES, NT>(buf, nvec, sh) : -INFINITY;
            float s = 0.f;
            if (m > -INFINITY && m < INFINITY)
                s = slice_sumexp<ES, NT>(buf, nvec, m, a.c_hi, a.c_lo, sh);
            if (tid == 0) {
                sh.part_m[par][r] = m;
                sh.part_s[par][r] = s;
            }
        }
        if (tid == 0)
            sh.part_flag[par] = timed_out ? 1 : 0;
        cluster.sync();

        // combine the C partials of each row in rank order, then decide
        if (warp == 0) {
            for (int r = 0; r < ng; ++r) {
                float mr = -INFINITY, sr = 0.f;
                int fr = 0;
                if (lane < a.C) {
                    const SvShared* rs = cluster.map_shared_rank(&sh, lane);
                    mr = rs->part_m[par][r];
                    sr = rs->part_s[par][r];
                    fr = rs->part_flag[par];
                }
                const float M = warp_max_nan<NT>(mr);
                double term = 0.0;
                if (lane < a.C && sr > 0.f && M > -INFINITY && M < INFINITY)
                    term = (double)sr * exp2(((double)mr - (double)M) * a.c_d);
#pragma unroll
                for (int o = 16; o; o >>= 1)
                    term += __shfl_down_sync(kFull, term, o);
                const int anyflag = __any_sync(kFull, fr != 0);
                if (lane == 0 && sh.state == kStateRun) {
                    const int i = g0 + r;
                    if (anyflag) {
                        sh.state = kStateError;
                        sh.code = SV_ERR_TIMEOUT;
                    } else if (!(M > -INFINITY && M < INFINITY)) {
                        sh.state = kStateError;
                        sh.code = SV_ERR_NONFINITE;
                    } else {
                        const double S = term;
                        sh.rs_m[i] = (float)((double)M / a.T_d);
                        sh.rs_s[i] = (float)S;
                        sh.ndec = i + 1;
                        if (i < K) {
                            const float qxf = sh.qx[i];
                            if (!(qxf >= 0.f && qxf < INFINITY)) {
                                sh.state = kStateError;
                                sh.code = SV_ERR_NONFINITE;
                            } else {
                                const double px = exp2(((double)sh.lx[i] - (double)M) * a.c_d) / S;
                                sh.pd[i] = (float)px;
                                if (!((double)sh.u[i] * (double)qxf < px)) {
                                    sh.state = kStateSample;
                                    sh.j = i;
                                    sh.mode = kModeResidual;
                                    sh.rowM = M;
                                    sh.rowS = S;
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
        __syncthreads();  // every thread is done with the staged rows
        load_group(g0, G < K + 1 - g0 ? G : K + 1 - g0);
    }

    // ---- corrected or bonus draw over row j ([P1]) ----
    if (sh.state == kStateSample) {
        const int j = sh.j;
        const unsigned char* buf = bufs + (size_t)(j - gcur) * a.rowbuf_bytes;
        const float* qrow = j < K ? a.q + ((int64_t)b * K + j) * V + v0 : nullptr;
        const float M = sh.rowM;
        const float inv_s = (float)(1.0 / sh.rowS);
        const double uK = (double)sh.u[K];
        const int ntiles = (nvec + NT - 1) / NT;
        int mode = sh.mode;
        int sp = 0;
        double S = 0.0, t = 0.0;
        double tots[sv::kMaxCluster];
        int lasts[sv::kMaxCluster];
        for (int round = 0; round < 2; ++round) {
            int last = -1;
            bool bad = false;
            for (int k = 0; k < ntiles; ++k) {
                const int vi = k * NT + tid;
                float ts = 0.f;
                if (vi < nvec) {
                    float w[E];
                    vec_weights<ES>(buf, vi, L, qrow, a.qvec, mode, M, a.c_hi, a.c_lo, inv_s, w,
                                    bad);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        ts += w[e];
                        if (w[e] > 0.f)
                            last = vi * E + e;
                    }
                }
                const float incl = warp_incl_scan(ts);
                if (lane == 31)
                    wt[k * NW + warp] = incl;
            }
            // block: any bad q, last positive entry, slice total
#pragma unroll
            for (int o = 16; o; o >>= 1)
                last = max(last, __shfl_xor_sync(kFull, last, o));
            if (lane == 0)
                sh.red_i[warp] = last;
            const int anybad = __syncthreads_or(bad);
            if (tid == 0) {
                int lb = -1;
                for (int w = 0; w < NW; ++w)
                    lb = max(lb, sh.red_i[w]);
                double tot = 0.0;
                for (int k = 0; k < ntiles; ++k)
                    for (int w = 0; w < NW; ++w)
                        tot += (double)wt[k * NW + w];
                sh.samp_tot[sp] = tot;
                sh.samp_last[sp] = lb >= 0 ? (int)(v0 + lb) : -1;
                sh.samp_bad[sp] = anybad;
            }
            cluster.sync();
            if (tid == 0) {
                int cbad = 0;
                S = 0.0;
                for (int c = 0; c < a.C; ++c) {
                    const SvShared* rs = cluster.map_shared_rank(&sh, c);
                    tots[c] = rs->samp_tot[sp];
                    lasts[c] = rs->samp_last[sp];
                    cbad |= rs->samp_bad[sp];
                    S += tots[c];
                }
                if (cbad) {
                    sh.state = kStateError;
                    sh.code = SV_ERR_NONFINITE;
                    sh.mode = -1;
                } else if (S == 0.0 && mode == kModeResidual) {
                    // max(0, p - q) vanished (rounding or an unnormalised q):
                    // draw from p_j itself with the same uniform
                    sh.mode = kModeTargetRow;
                } else {
                    sh.mode = -1;  // done
                    t = uK * S;
                    int owner = -1;
                    double run = 0.0;
                    for (int c = 0; c < a.C; ++c) {
                        if (run + tots[c] > t) {
                            owner = c;
                            break;
                        }
                        run += tots[c];
                    }
                    sh.tok = -1;
                    if (owner < 0) {
                        // rounding left t at or past the total: last positive entry
                        for (int c = a.C - 1; c >= 0; --c)
                            if (lasts[c] >= 0) {
                                sh.tok = lasts[c];
                                break;
                            }
                        owner = 0;
                    }
                    sh.owner = owner;
                    sh.loc_rem = t - run;
                }
            }
            __syncthreads();
            if (sh.mode != kModeTargetRow)
                break;
            mode = kModeTargetRow;
            sp ^= 1;
        }

        if (sh.state == kStateSample && rank == sh.owner) {
            // locate the crossing inside this CTA's slice: tile, then warp
            if (tid == 0 && sh.tok < 0) {
                const double rem = sh.loc_rem;
                double acc = 0.0;
                int kk = -1, ww = -1;
                for (int k = 0; k < ntiles && kk < 0; ++k) {
                    double tk = 0.0;
                    for (int w = 0; w < NW; ++w)
                        tk += (double)wt[k * NW + w];
                    if (acc + tk > rem) {
                        for (int w = 0; w < NW; ++w) {
                            const double tw = (double)wt[k * NW + w];
                            if (acc + tw > rem) {
                                kk = k;
                                ww = w;
                                break;
                            }
                            acc += tw;
                        }
                        if (kk < 0)
                            break;  // rounding: no warp crosses inside the tile
                    } else {
                        acc += tk;
                    }
                }
                if (kk < 0) {
                    sh.tok = sh.samp_last[sp];
                } else {
                    sh.loc_tile = kk;
                    sh.loc_warp = ww;
                    sh.loc_rem = rem - acc;
                }
            }
            __syncthreads();
            if (sh.tok < 0 && warp == sh.loc_warp) {
                // this warp re-derives the same weights and scan, then finds
                // the lane and the entry where the running sum passes the rest
                const double rem = sh.loc_rem;
                const int vi = sh.loc_tile * NT + tid;
                float w[E];
                float ts = 0.f;
                bool dummy = false;
                if (vi < nvec) {
                    vec_weights<ES>(buf, vi, L, qrow, a.qvec, mode, M, a.c_hi, a.c_lo, inv_s, w,
                                    dummy);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        ts += w[e];
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        w[e] = 0.f;
                }
                const float incl = warp_incl_scan(ts);
                float excl = __shfl_up_sync(kFull, incl, 1);
                if (lane == 0)
                    excl = 0.f;
                const unsigned cross = __ballot_sync(kFull, (double)incl > rem);
                const unsigned pos = __ballot_sync(kFull, ts > 0.f);
                int pick = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : -1);
                if (lane == pick) {
                    int e_hit = -1, e_last = -1;
                    double acc = (double)excl;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if (w[e] > 0.f)
                            e_last = e;
                        acc += (double)w[e];
                        if (e_hit < 0 && cross && acc > rem)
                            e_hit = e;
                    }
                    const int e = e_hit >= 0 ? e_hit : e_last;
                    sh.tok = e >= 0 ? (int)(v0 + (int64_t)vi * E + e) : sh.samp_last[sp];
                }
                __syncwarp();
                if (lane == 0 && pick < 0)
                    sh.tok = sh.samp_last[sp];
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
    return spec_verify_plan_for(ctx->num_sms, ctx->smem_optin, ctx->max_cluster, B, K, V, dtype,
                                ctx->ovr_cluster, ctx->ovr_group, ctx->ovr_threads, plan);
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
    args.bulk = plan.bulk_copy && aligned(logits, 16) ? 1 : 0;
    args.qvec = (V % 4 == 0) && q && aligned(q, 16) ? 1 : 0;
    args.T_d = (double)T;
    args.c_d = 1.4426950408889634074 / args.T_d;  // log2(e) / T
    args.c_hi = (float)args.c_d;
    args.c_lo = (float)(args.c_d - (double)args.c_hi);
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
