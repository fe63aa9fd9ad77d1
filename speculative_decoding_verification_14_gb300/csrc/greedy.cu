// greedy.cu -- greedy verification (the verify step in the limit T -> 0) for
// sm_103a.
//
// As T falls, the softmax of l/T in [P1]'s loop puts all of its mass on the
// largest logit, so each target row becomes one-hot at a_i = argmax_v l[b,i,v]
// (the lowest id among equal maxima).  The test u*q(x) < p(x) then accepts
// exactly when x_i = a_i, the residual max(0, p_j - q_j) is positive only at
// a_j, and the bonus row yields a_K: the step needs the target rows alone, no
// draft probabilities and no uniforms.  Like [P1]'s loop it reads the rows in
// order and stops at the first rejection.
//
// [P1] reactapp.top, "Speculative decoding and early exit: speeding up
//      autoregressive decode", section "Speculative decoding: draft first,
//      then verify" (the conceptual loop and its temperature).
//
// Design: a thread-block cluster of C CTAs per sequence, CTA r owning a
// vocabulary slice of every row and each warp a stretch of that slice.  Lanes
// stream 16-byte vectors (eight deep per lane) with non-allocating loads and
// keep the largest value and the first entry holding it (found from the
// registers in the rare step where the maximum grows).  Each warp pushes its
// partial (value, lowest index, bad-value flag) into a slot of every CTA of
// the cluster with st.async, counted on that CTA's mbarrier; every warp then
// merges all partials itself and reaches the same decision, so a row costs no
// CTA or cluster barrier.
#include <cuda_runtime.h>
#include <cooperative_groups.h>

#include <cstdint>
#include <cstring>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kNT = 128;                  // threads per CTA
constexpr int kNW = kNT / 32;
constexpr int kDepth = sv::kGreedyDepth;  // 16-byte loads in flight per lane
constexpr int kNoIndex = 0x7fffffff;

struct GArgs {
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
    int B, K, C, vec;
    unsigned long long wait_ns;
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

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

// Entry e of a 16-byte vector as a float (bf16 widens exactly).
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

// Largest entry of a vector, NaN if any entry is NaN.
template <int ES>
__device__ __forceinline__ float vec_max(const uint4& v) {
    if constexpr (ES == 4) {
        return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                        fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    } else {
        const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
        return fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
}

__device__ __forceinline__ float load_entry(const void* base, int es, int64_t idx) {
    if (es == 4)
        return __ldg(static_cast<const float*>(base) + idx);
    const uint16_t h = __ldg(static_cast<const unsigned short*>(base) + idx);
    return __uint_as_float((uint32_t)h << 16);
}

// (value, index) of the better partial: larger value, then lower index.
__device__ __forceinline__ void better(float& v, int& i, float ov, int oi) {
    if (ov > v || (ov == v && oi < i)) {
        v = ov;
        i = oi;
    }
}

__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
    for (int s = 16; s; s >>= 1)
        better(v, i, __shfl_xor_sync(kFull, v, s), __shfl_xor_sync(kFull, i, s));
}

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

// Wait for phase `parity` of `bar`, sleeping between polls; false after
// `limit_ns` (the partials never came).
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

// 16 bytes into the same shared-memory slot of cluster CTA `rank`, counted on
// that CTA's barrier `bar` (same offset) as complete_tx.
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

template <int ES>
__global__ void __launch_bounds__(kNT, 8) sv_greedy_kernel(const __grid_constant__ GArgs a) {
    constexpr int E = 16 / ES;  // entries per 16-byte vector
    constexpr uint32_t kPad = ES == 2 ? 0xff80ff80u : 0xff800000u;  // -inf entries past the stretch
    constexpr int kPer = (sv::kMaxCluster * kNW + 31) / 32;           // partials per lane, at most
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)a.C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, C = a.C;
    const int P = C * kNW;  // partials per row: every warp of the cluster
    const int64_t V = a.V;

    // part[parity][rank * kNW + warp] is pushed by that warp of every CTA;
    // xbar[parity] counts the bytes (one phase per row of that parity)
    __shared__ __align__(16) float4 part[2][sv::kMaxCluster * kNW];
    __shared__ __align__(8) unsigned long long xbar[2];
    __shared__ int xs[sv::kMaxK];

    const int64_t v0 = (int64_t)rank * a.slice;
    const int64_t L = v0 < V ? (V - v0 < a.slice ? V - v0 : a.slice) : 0;
    const int64_t row0 = (int64_t)b * (K + 1);

    if (tid == 0) {
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < K)
        xs[tid] = a.tokens[(int64_t)b * K + tid];
    __syncthreads();
    // every CTA's barriers are initialised before anyone pushes into them
    cluster_arrive();
    bool ready = false;
    int state = SV_OK;
    if (__any_sync(kFull, lane < K && (xs[lane] < 0 || (int64_t)xs[lane] >= V)))
        state = SV_ERR_TOKEN_RANGE;

    // this warp's stretch: vectors [w0, w1) of the slice (or entries, on the
    // element path)
    const int64_t units = a.vec ? L / E : L;
    const int64_t per_w = (units + kNW - 1) / kNW;
    const int64_t w0 = per_w * warp < units ? per_w * warp : units;
    const int64_t w1 = w0 + per_w < units ? w0 + per_w : units;

    int j = -1, tok = -1;
    for (int i = 0; i <= K && state == SV_OK; ++i) {
        const int par = i & 1;
        const uint32_t phase = (uint32_t)(i >> 1) & 1u;
        if (tid == 0)  // this row's partials, from every warp of the cluster
            mbar_expect(&xbar[par], (uint32_t)(P * 16));
        const unsigned char* row =
            static_cast<const unsigned char*>(a.logits) + ((row0 + i) * V + v0) * ES;
        float best = -INFINITY;
        int bidx = kNoIndex;
        bool bad = false;
        if (a.vec) {
            const uint4* rp = reinterpret_cast<const uint4*>(row);
            for (int64_t base = w0; base < w1; base += 32 * kDepth) {
                uint4 r[kDepth];
#pragma unroll
                for (int k = 0; k < kDepth; ++k) {
                    const int64_t idx = base + k * 32 + lane;
                    r[k] = idx < w1 ? ld_stream(rp + idx) : make_uint4(kPad, kPad, kPad, kPad);
                }
#pragma unroll
                for (int k = 0; k < kDepth; ++k) {
                    const float m = vec_max<ES>(r[k]);
                    if (!(m <= best)) {  // larger, or NaN (rare after the first vectors)
                        if (m != m) {
                            bad = true;
                        } else {  // the first entry of this vector holding m
                            int e = E - 1;
#pragma unroll
                            for (int t = E - 1; t >= 0; --t)
                                if (vec_entry<ES>(r[k], t) == m)
                                    e = t;
                            best = m;
                            bidx = (int)(v0 + (base + k * 32 + lane) * E + e);
                        }
                    }
                }
            }
        } else {
            for (int64_t e = w0 + lane; e < w1; e += 32) {
                const float l = load_entry(a.logits, ES, (row0 + i) * V + v0 + e);
                if (l != l)
                    bad = true;
                else if (l > best) {
                    best = l;
                    bidx = (int)(v0 + e);
                }
            }
        }
        if (best == INFINITY)
            bad = true;
        warp_best(best, bidx);
        bad = __any_sync(kFull, bad);
        if (!ready) {
            cluster_wait();
            ready = true;
        }
        if (lane < C)
            push_v4(&part[par][rank * kNW + warp], &xbar[par], (uint32_t)lane,
                    make_float4(best, __int_as_float(bidx), bad ? 1.f : 0.f, 0.f));
        // every warp merges the P partials itself and reaches the same decision
        // (one outcome for the whole warp, even when the wait runs out)
        if (!__all_sync(kFull, mbar_wait_limited(&xbar[par], phase, a.wait_ns))) {
            state = SV_ERR_TIMEOUT;
            break;
        }
        float v = -INFINITY;
        int ix = kNoIndex;
        bool any_bad = false;
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
            const int p = lane + 32 * t;
            if (p < P) {
                const float4 q = part[par][p];
                better(v, ix, q.x, __float_as_int(q.y));
                any_bad |= q.z != 0.f;
            }
        }
        warp_best(v, ix);
        any_bad = __any_sync(kFull, any_bad);
        if (any_bad || !(v > -INFINITY)) {
            state = SV_ERR_NONFINITE;
            break;
        }
        if (a.row_argmax && rank == 0 && tid == 0)
            a.row_argmax[row0 + i] = ix;
        if (i < K && xs[i] == ix)
            continue;
        j = i;
        tok = ix;
        break;
    }

    if (rank == 0 && warp == 0) {
        const bool err = state != SV_OK;
        for (int i = lane; i <= K; i += 32) {
            int t = -1;
            if (!err)
                t = i < j ? xs[i] : (i == j ? tok : -1);
            a.out_tokens[row0 + i] = t;
            if (i < K)
                a.accept_mask[(int64_t)b * K + i] = (!err && i < j) ? 1 : 0;
            if (a.row_argmax && (err || i > j))
                a.row_argmax[row0 + i] = -1;
        }
        if (lane == 0) {
            a.accept_len[b] = err ? 0 : j + 1;
            if (a.status)
                a.status[b] = state;
            if (err)
                atomicOr(a.err_word, 1u << state);
            if (a.al_hist)
                atomicAdd(a.al_hist + (err ? 0 : j + 1), 1u);
        }
    }
    // no CTA leaves while a push into it may still be on its way
    if (!ready)
        cluster_wait();
    cluster_arrive();
    cluster_wait();
}

// Self-test of the bounded wait above (the routine every wait of this
// kernel goes through): one thread waits on a barrier of its own.  With
// `arrive` the thread first completes the barrier's phase 0, so the wait must
// succeed at once; without it nothing ever arrives, so the wait must give up
// once limit_ns have passed.  Nothing is in flight when it returns.
__device__ unsigned long long sv_wait_selftest_out[2];  // completed, elapsed ns

__global__ void sv_wait_selftest_kernel(unsigned long long limit_ns, int arrive) {
    __shared__ __align__(8) unsigned long long bar;
    mbar_init(&bar, 1);
    if (arrive)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&bar)) : "memory");
    const unsigned long long t0 = now_ns();
    const bool ok = mbar_wait_limited(&bar, 0, limit_ns);
    sv_wait_selftest_out[0] = ok ? 1ull : 0ull;
    sv_wait_selftest_out[1] = now_ns() - t0;
}

}  // namespace

extern "C" int spec_verify_selftest_wait(int device, unsigned long long limit_ns, int arrive,
                                         int* completed, unsigned long long* elapsed_ns) {
    if (!completed || !elapsed_ns || limit_ns > 2000000000ull)
        return SV_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    sv_wait_selftest_kernel<<<1, 1>>>(limit_ns, arrive ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(0);
    unsigned long long h[2] = {0, 0};
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbol(h, sv_wait_selftest_out, sizeof h);
    (void)cudaSetDevice(prev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return SV_ERR_CUDA;
    }
    *completed = (int)h[0];
    *elapsed_ns = h[1];
    return SV_OK;
}

namespace sv {

int greedy_set_attributes() {
    const void* fns[2] = {(const void*)sv_greedy_kernel<2>, (const void*)sv_greedy_kernel<4>};
    for (const void* f : fns)
        if (cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return 1;
        }
    return 0;
}

int greedy_launch(const GreedyLaunch& g, void* stream) {
    GArgs a;
    std::memset(&a, 0, sizeof a);
    a.logits = g.logits;
    a.tokens = g.tokens;
    a.accept_len = g.accept_len;
    a.out_tokens = g.out_tokens;
    a.accept_mask = g.accept_mask;
    a.row_argmax = g.row_argmax;
    a.status = g.status;
    a.err_word = g.err_word;
    a.al_hist = g.al_hist;
    a.V = g.V;
    a.slice = g.slice;
    a.B = g.B;
    a.K = g.K;
    a.C = g.C;
    a.vec = g.vec;
    a.wait_ns = g.wait_ns;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)((int64_t)g.B * g.C), 1, 1);
    cfg.blockDim = dim3(kNT, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)g.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = g.es == 2 ? cudaLaunchKernelEx(&cfg, sv_greedy_kernel<2>, a)
                                    : cudaLaunchKernelEx(&cfg, sv_greedy_kernel<4>, a);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return 0;
}

}  // namespace sv
