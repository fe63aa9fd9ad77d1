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
// keep the largest vector maximum and the vector that first reached it; the
// entry index is recovered at the end of the row by re-reading that one
// vector.  Warp, CTA and cluster partials (value, lowest index, bad-value
// flag) meet through shared memory and one cluster barrier per row; every CTA
// takes the same decision from the same data.
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

__device__ __forceinline__ float4 ld_cluster_v4(const void* local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(local)), "r"(rank));
    float4 r;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "r"(a)
                 : "memory");
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int ES>
__global__ void __launch_bounds__(kNT, 8) sv_greedy_kernel(const __grid_constant__ GArgs a) {
    constexpr int E = 16 / ES;  // entries per 16-byte vector
    constexpr uint32_t kPad = ES == 2 ? 0xff80ff80u : 0xff800000u;  // -inf entries past the stretch
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / (unsigned)a.C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, C = a.C;
    const int64_t V = a.V;

    __shared__ float4 wpart[kNW];          // per warp: (value, index bits, bad, 0)
    __shared__ __align__(16) float4 cpart[2];  // this CTA's partial, by row parity
    __shared__ int dec[2];                 // (a_i, state) of the row just decided
    __shared__ int xs[sv::kMaxK];

    const int64_t v0 = (int64_t)rank * a.slice;
    const int64_t L = v0 < V ? (V - v0 < a.slice ? V - v0 : a.slice) : 0;
    const int64_t row0 = (int64_t)b * (K + 1);

    if (tid < K)
        xs[tid] = a.tokens[(int64_t)b * K + tid];
    __syncthreads();
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
        const unsigned char* row =
            static_cast<const unsigned char*>(a.logits) + ((row0 + i) * V + v0) * ES;
        float best = -INFINITY;
        int bidx = kNoIndex;
        bool bad = false;
        if (a.vec) {
            const uint4* rp = reinterpret_cast<const uint4*>(row);
            int64_t bvec = -1;
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
                    if (!(m <= best)) {  // larger, or NaN
                        if (m != m) {
                            bad = true;
                        } else {
                            best = m;
                            bvec = base + k * 32 + lane;
                        }
                    }
                }
            }
            if (bvec >= 0 && best > -INFINITY) {  // the first entry of that vector holding best
                const uint4 r = ld_stream(rp + bvec);
                int e = E - 1;
#pragma unroll
                for (int t = E - 1; t >= 0; --t)
                    if (vec_entry<ES>(r, t) == best)
                        e = t;
                bidx = (int)(v0 + bvec * E + e);
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
        const int par = i & 1;
        if (lane == 0)
            wpart[warp] = make_float4(best, __int_as_float(bidx), bad ? 1.f : 0.f, 0.f);
        __syncthreads();
        if (warp == 0) {
            float v = -INFINITY;
            int ix = kNoIndex;
            float bd = 0.f;
            if (lane < kNW) {
                const float4 p = wpart[lane];
                v = p.x;
                ix = __float_as_int(p.y);
                bd = p.z;
            }
            warp_best(v, ix);
            const bool any_bad = __any_sync(kFull, bd != 0.f);
            if (lane == 0)
                cpart[par] = make_float4(v, __int_as_float(ix), any_bad ? 1.f : 0.f, 0.f);
        }
        cluster_sync_all();  // every CTA's partial of row i is in place
        if (warp == 0) {
            float v = -INFINITY;
            int ix = kNoIndex;
            float bd = 0.f;
            if (lane < C) {
                const float4 p = ld_cluster_v4(&cpart[par], (uint32_t)lane);
                v = p.x;
                ix = __float_as_int(p.y);
                bd = p.z;
            }
            warp_best(v, ix);
            const bool any_bad = __any_sync(kFull, bd != 0.f);
            if (lane == 0) {
                dec[0] = ix;
                dec[1] = (any_bad || !(v > -INFINITY)) ? SV_ERR_NONFINITE : SV_OK;
            }
        }
        __syncthreads();
        const int ai = dec[0];
        state = dec[1];
        __syncthreads();  // dec is rewritten by the next row
        if (state != SV_OK)
            break;
        if (a.row_argmax && rank == 0 && tid == 0)
            a.row_argmax[row0 + i] = ai;
        if (i < K && xs[i] == ai)
            continue;
        j = i;
        tok = ai;
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
    // no CTA leaves while another may still read its partials
    cluster_sync_all();
}

}  // namespace

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
