// sdm_gwr.cu -- GWR, the token gather of the write side of the chunked sparse-delta-memory
// backward, and its C entry point sdm_gwr (include/sdm.h).
//
// Arithmetic (sparse-delta-memory 2.0.0, pa_dc_cuda.py: module docstring, "GWR", and its GWR kernel),
// per chunk c = ti * P + p and valid token t (padding tokens get zeros):
//   d_delta_v[c, t] = acc, acc = 0; acc = fmaf(write_w[c, t, n], grad[p*S + k_idx[c, t, n]], acc)
//                     over the write lanes n = 0 .. W-1 in order;
//   d_k_pd[c, t, n] = <dv[c*C + t], grad[p*S + k_idx[c, t, n]]>,
// the dot summed like every dot of the backward here (per lane an fmaf chain over its 4 columns of a
// 128-column slice, the 32 lane partials in one fixed lane tree, slices added in order from 0).
//
// GB300 design: one launch per step, one warp per token. The grad rows of 16 write lanes are in flight
// at once (a lane's 4 columns of each, kept in the storage type); the same registers feed the
// gather's fmaf chain and the 16 dots, which are reduced across the lanes together (transposed), lane
// n storing d_k_pd of lane n. Rows wider than 128 columns take their slices one after the other; a
// token's dot sums are then carried in d_k_pd between slices by the lane that stores them.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "sdm_checks.cuh"
#include "sdm_internal.cuh"
#include "sdm_rows.cuh"

namespace sdm {
namespace {

using namespace rows;

constexpr int kGwrThreads = 256;
constexpr int kGwrWarps = kGwrThreads / 32;

struct GWRArgs {
    const int32_t* k_idx;      // [N, C, W]
    const float* write_w;      // [N, C, W]
    const void* dv;            // [N * C, hd] dv type
    const void* grad;          // [P * S, hd] grad type (read only)
    float* d_delta_v;          // [N, C, hd]
    float* d_k_pd;             // [N, C, W]
    uint32_t* status;          // nullable
    int P, C, W, hd, nsl, groups;
    int valid;                 // valid tokens of this step's chunks
    int64_t S, c0;
};

template <typename GradT, typename DvT>
__global__ void __launch_bounds__(kGwrThreads) gwr_kernel(const GWRArgs a) {
    // launched as a programmatic dependent of the kernel before it (the previous step's kernel, or any
    // kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cl = static_cast<int>(blockIdx.x / a.groups);
    const int tg = static_cast<int>(blockIdx.x - static_cast<int64_t>(cl) * a.groups);
    const int t = tg * kGwrWarps + warp;
    if (t >= a.C) return;   // warp-uniform
    const int64_t c = a.c0 + cl;
    const int hd = a.hd, W = a.W;
    const bool tvalid = t < a.valid;
    const int64_t tok = c * a.C + t;
    const GradT* const grad = static_cast<const GradT*>(a.grad) + static_cast<int64_t>(cl) * a.S * hd;
    const DvT* const dvrow = static_cast<const DvT*>(a.dv) + tok * hd;
    const int32_t* const ki = a.k_idx + tok * W;
    const float* const wi = a.write_w + tok * W;
    float* const pd = a.d_k_pd + tok * W;
    float* const out = a.d_delta_v + tok * hd;
    uint32_t bad = 0;
    for (int sl = 0; sl < a.nsl; ++sl) {
        const int col = sl * 128 + lane * 4;
        const bool on = col < hd;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (on && tvalid) ld4(dvrow + col, x);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int e0 = 0; e0 < W; e0 += 16) {
            // lane e < 16: the slot and weight of write lane e0 + e (slot -1: no row)
            int32_t myslot = -1;
            float myw = 0.f;
            if (tvalid && lane < 16 && e0 + lane < W) {
                myslot = __ldg(ki + e0 + lane);
                myw = __ldg(wi + e0 + lane);
                if (myslot < 0 || static_cast<int64_t>(myslot) >= a.S) {
                    myslot = -1;
                    bad = 1u;
                }
            }
            // the 16 lanes' grad rows, all in flight: every load is unconditional (a lane without a
            // row reads row 0 / column 0 of the stream and drops the value), so none waits on a branch
            const uint32_t hasrow = __ballot_sync(kFull, myslot >= 0);
            const int ccol = on ? col : 0;
            Raw4<GradT> g[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int32_t s = __shfl_sync(kFull, myslot, e);
                g[e].ld(grad + static_cast<int64_t>(s < 0 ? 0 : s) * hd + ccol);
            }
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float we = __shfl_sync(kFull, myw, e);
                float gf[4];
                g[e].get(gf);
                const bool use = ((hasrow >> e) & 1u) && on;
#pragma unroll
                for (int i = 0; i < 4; ++i) gf[i] = use ? gf[i] : 0.f;
                if ((hasrow >> e) & 1u) {   // warp-uniform
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(we, gf[i], acc[i]);
                }
                v[e] = dot4(x, gf);
            }
            const float r = tsum16(v, lane);   // lane l: write lane e0 + (l & 15)
            if (lane < 16 && e0 + lane < W) pd[e0 + lane] = (sl == 0 ? 0.f : pd[e0 + lane]) + r;
        }
        if (on) st4(out + col, acc);
    }
    if (__any_sync(kFull, bad != 0) && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

// Rows of at most 128 columns and at most 16 write lanes (one slice, one block of lanes): the same
// arithmetic as gwr_kernel, with a grid of resident warps only, each looping over tokens; the next
// token's ids, weights and dv row load while the current token's grad rows are in flight.
template <typename GradT, typename DvT>
__global__ void __launch_bounds__(kGwrThreads) gwr_loop_kernel(const GWRArgs a, int total_warps) {
    // launched as a programmatic dependent of the kernel before it (the previous step's kernel, or any
    // kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int ntok = a.P * a.C;
    int it = blockIdx.x * kGwrWarps + (threadIdx.x >> 5);
    if (it >= ntok) return;   // warp-uniform
    const int hd = a.hd, W = a.W;
    const int col = lane * 4;
    const bool on = col < hd;
    const int ccol = on ? col : 0;
    uint32_t bad = 0;
    // a token's ids, weights (lanes < W) and dv row
    auto fetch = [&](int i, int32_t& slot, float& wt, float (&x)[4]) {
        const int cl = i / a.C, t = i - cl * a.C;
        const int64_t tok = (a.c0 + cl) * a.C + t;
        slot = -1;
        wt = 0.f;
        x[0] = x[1] = x[2] = x[3] = 0.f;
        if (t < a.valid) {
            if (lane < W) {
                slot = __ldg(a.k_idx + tok * W + lane);
                wt = __ldg(a.write_w + tok * W + lane);
                if (slot < 0 || static_cast<int64_t>(slot) >= a.S) {
                    slot = -1;
                    bad = 1u;
                }
            }
            if (on) ld4(static_cast<const DvT*>(a.dv) + tok * hd + col, x);
        }
    };
    int32_t myslot;
    float myw, x[4];
    fetch(it, myslot, myw, x);
    for (;;) {
        const int cl = it / a.C, t = it - cl * a.C;
        const int64_t tok = (a.c0 + cl) * a.C + t;
        const GradT* const grad = static_cast<const GradT*>(a.grad) + static_cast<int64_t>(cl) * a.S * hd;
        const uint32_t hasrow = __ballot_sync(kFull, myslot >= 0);
        Raw4<GradT> g[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int32_t s = __shfl_sync(kFull, myslot, e);
            g[e].ld(grad + static_cast<int64_t>(s < 0 ? 0 : s) * hd + ccol);
        }
        const int nit = it + total_warps;
        int32_t nslot = -1;
        float nw = 0.f, nx[4] = {0.f, 0.f, 0.f, 0.f};
        if (nit < ntok) fetch(nit, nslot, nw, nx);
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float we = __shfl_sync(kFull, myw, e);
            float gf[4];
            g[e].get(gf);
            const bool use = ((hasrow >> e) & 1u) && on;
#pragma unroll
            for (int i = 0; i < 4; ++i) gf[i] = use ? gf[i] : 0.f;
            if ((hasrow >> e) & 1u) {   // warp-uniform
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = fmaf(we, gf[i], acc[i]);
            }
            v[e] = dot4(x, gf);
        }
        const float r = tsum16(v, lane);
        if (lane < W) a.d_k_pd[tok * W + lane] = 0.f + r;
        if (on) st4(a.d_delta_v + tok * hd + col, acc);
        if (nit >= ntok) break;
        it = nit;
        myslot = nslot;
        myw = nw;
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = nx[i];
    }
    if (__any_sync(kFull, bad != 0) && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

template <typename GradT, typename DvT>
cudaError_t launch_gd(const GWRArgs& a, cudaStream_t stream) {
    if (a.nsl == 1 && a.W <= 16) {
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gwr_loop_kernel<GradT, DvT>, kGwrThreads, 0);
        if (e != cudaSuccess) return e;
        const int ntok = a.P * a.C;
        const int blocks = std::max(1, std::min((ntok + kGwrWarps - 1) / kGwrWarps, sms * std::max(per_sm, 1)));
        return launch_dependent(gwr_loop_kernel<GradT, DvT>, dim3(blocks), dim3(kGwrThreads), 0, stream, a,
                                blocks * kGwrWarps);
    }
    return launch_dependent(gwr_kernel<GradT, DvT>, dim3(static_cast<unsigned>(a.P) * a.groups), dim3(kGwrThreads), 0,
                            stream, a);
}

template <typename GradT>
cudaError_t launch_g(const GWRArgs& a, int dv_bf16, cudaStream_t stream) {
    return dv_bf16 ? launch_gd<GradT, __nv_bfloat16>(a, stream) : launch_gd<GradT, float>(a, stream);
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" sdm_status sdm_gwr(const sdm_shape* shape, int32_t grad_dtype, const int32_t* k_idx, const float* write_w,
                              const void* dv, const void* grad, float* d_delta_v, float* d_k_pd, int64_t step_begin,
                              int64_t step_end, uint32_t* status, sdm_stream_t stream) {
    const void* const ptrs[] = {k_idx, write_w, dv, grad, d_delta_v, d_k_pd};
    const sdm_status st = checks::check_backward(shape, grad_dtype, step_begin, step_end, ptrs);
    if (st != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    GWRArgs a;
    memset(&a, 0, sizeof(a));
    a.k_idx = k_idx;
    a.write_w = write_w;
    a.dv = dv;
    a.grad = grad;
    a.d_delta_v = d_delta_v;
    a.d_k_pd = d_k_pd;
    a.status = status;
    a.P = shape->P;
    a.C = shape->C;
    a.W = shape->W;
    a.hd = shape->hd;
    a.nsl = (shape->hd + 127) / 128;
    a.groups = (shape->C + kGwrWarps - 1) / kGwrWarps;
    a.S = shape->S;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    for (int64_t ti = step_end - 1; ti >= step_begin; --ti) {   // last step first, like the backward
        a.c0 = ti * a.P;
        a.valid = ti == shape->steps - 1 ? shape->valid_last : shape->C;
        const cudaError_t e = grad_dtype == SDM_BF16 ? launch_g<__nv_bfloat16>(a, shape->dv_dtype == SDM_BF16, cs)
                                                     : launch_g<float>(a, shape->dv_dtype == SDM_BF16, cs);
        if (e != cudaSuccess) return SDM_ERR_CUDA;
    }
    return SDM_OK;
}
