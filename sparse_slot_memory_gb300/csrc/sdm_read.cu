// sdm_read.cu -- the forward's read-side token gather of the chunked sparse-delta-memory recurrence
// and its C entry point sdm_read (include/sdm.h).
//
// Arithmetic (sparse-delta-memory 2.0.0: mover_fx_cuda.py, fx_fwd_steps -- each step's gather before
// its dual matmul and DW; the weighted read whose vector-Jacobian product in q_w is the GDS dot of
// mover_da2_cuda.py's module docstring, d_q_w[t, r] = <gr[t], bank[slot]>; the token_gather form of
// GWR's d_delta_v, pa_dc_cuda.py's module docstring), per chunk c = ti * P + p and valid token t
// (padding tokens get zeros):
//   y[c, t] = acc, acc = 0; acc = fmaf(q_w[c, t, r], bank[p*S + q_idx[c, t, r]], acc)
//             over the read lanes r = 0 .. R-1 in order (a lane whose id is outside [0, S) adds nothing).
//
// GB300 design: a grid of resident warps (as many as the SMs hold), each looping over (token, 128-column
// slice) units, launched as a programmatic dependent of the previous kernel (its launch latency is
// hidden). A unit's 16 read rows are all in flight at once (each lane its 4 columns, kept in the
// storage type), then summed in lane order; the next unit's ids and weights load while the current
// unit's rows are in flight. HBM-bound: per token R ids and weights, one bank row per valid read lane,
// one f32 output row.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "sdm_checks.cuh"
#include "sdm_internal.cuh"
#include "sdm_rows.cuh"

namespace sdm {
namespace {

using namespace rows;

constexpr int kReadThreads = 256;
constexpr int kReadWarps = kReadThreads / 32;

struct ReadArgs {
    const int32_t* q_idx;   // [N, C, R]
    const void* q_w;        // [N, C, R] value type
    const void* bank;       // [P * S, hd] bank type (read only)
    float* y;               // [N, C, hd]
    uint32_t* status;       // nullable
    int P, C, R, hd, nsl, valid_last;
    int64_t S, steps, c0;
    int64_t units;          // chunks of the range * C * nsl
};

template <typename BankT, typename WT>
// bf16 banks: 4 blocks of 8 warps per SM at 64 registers (measured 10.2 -> 9.9 us per step on the large
// workload against 3 blocks at 80); f32 banks keep 2 (108 registers: 4 per lane per row in flight)
__global__ void __launch_bounds__(kReadThreads, sizeof(BankT) == 2 ? 4 : 2) read_kernel(const ReadArgs a, int64_t total_warps) {
    // launched as a programmatic dependent of the kernel before it (the previous step's read or DW, or
    // any kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    int64_t u = static_cast<int64_t>(blockIdx.x) * kReadWarps + (threadIdx.x >> 5);
    if (u >= a.units) return;   // warp-uniform
    const int per_chunk = a.C * a.nsl;
    uint32_t bad = 0;
    // a unit's token, slice and (lanes < 16) the ids and weights of read lanes r0 + lane
    auto fetch = [&](int64_t uu, int r0, int32_t& slot, float& wt) {
        const int64_t cl = uu / per_chunk;
        const int rest = static_cast<int>(uu - cl * per_chunk);
        const int t = rest / a.nsl;
        const int64_t c = a.c0 + cl;
        const int V = c / a.P == a.steps - 1 ? a.valid_last : a.C;
        slot = -1;
        wt = 0.f;
        if (t < V && lane < 16 && r0 + lane < a.R) {
            const int64_t e = (c * a.C + t) * a.R + r0 + lane;
            slot = __ldg(a.q_idx + e);
            wt = widen(__ldg(static_cast<const WT*>(a.q_w) + e));
            if (slot < 0 || static_cast<int64_t>(slot) >= a.S) {
                slot = -1;
                bad = 1u;
            }
        }
    };
    int32_t myslot;
    float myw;
    fetch(u, 0, myslot, myw);
    for (;;) {
        const int64_t cl = u / per_chunk;
        const int rest = static_cast<int>(u - cl * per_chunk);
        const int t = rest / a.nsl, sl = rest - t * a.nsl;
        const int64_t c = a.c0 + cl;
        const int64_t p = c % a.P;
        const int col = sl * 128 + lane * 4;
        const bool on = col < a.hd;
        const int ccol = on ? col : 0;
        const BankT* const bank = static_cast<const BankT*>(a.bank) + p * a.S * a.hd;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r0 = 0;;) {
            // the 16 lanes' rows, all in flight: every load is unconditional (a lane without a row
            // reads row 0 / column 0 of the stream and drops the value), so none waits on a branch
            const uint32_t hasrow = __ballot_sync(kFull, myslot >= 0);
            Raw4<BankT> g[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int32_t s = __shfl_sync(kFull, myslot, e);
                g[e].ld(bank + static_cast<int64_t>(s < 0 ? 0 : s) * a.hd + ccol);
            }
            // the next ids and weights: this unit's next 16 lanes, else the next unit's first 16
            const int nr0 = r0 + 16;
            const int64_t nu = nr0 < a.R ? u : u + total_warps;
            int32_t nslot = -1;
            float nw = 0.f;
            if (nu < a.units) fetch(nu, nr0 < a.R ? nr0 : 0, nslot, nw);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float we = __shfl_sync(kFull, myw, e);
                float gf[4];
                g[e].get(gf);
                if ((hasrow >> e) & 1u) {   // warp-uniform
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(we, gf[i], acc[i]);
                }
            }
            myslot = nslot;
            myw = nw;
            if (nr0 >= a.R) break;
            r0 = nr0;
        }
        if (on) st4(a.y + (c * a.C + t) * static_cast<int64_t>(a.hd) + col, acc);
        u += total_warps;
        if (u >= a.units) break;
    }
    if (__any_sync(kFull, bad != 0) && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

template <typename BankT, typename WT>
cudaError_t launch_r(const ReadArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, read_kernel<BankT, WT>, kReadThreads, 0);
    if (e != cudaSuccess) return e;
    const int64_t want = (a.units + kReadWarps - 1) / kReadWarps;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(sms) * std::max(per_sm, 1)));
    return launch_dependent(read_kernel<BankT, WT>, dim3(static_cast<unsigned>(blocks)), dim3(kReadThreads), 0, stream, a,
                            static_cast<int64_t>(blocks * kReadWarps));
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" sdm_status sdm_read(const sdm_shape* shape, const int32_t* q_idx, const void* q_w, const void* bank,
                               float* y, int64_t step_begin, int64_t step_end, uint32_t* status,
                               sdm_stream_t stream) {
    sdm_status st = checks::check_shape(shape);
    if (st != SDM_OK) return st;
    if (step_begin < 0 || step_end > shape->steps || step_begin > step_end) return SDM_ERR_ARG;
    if (q_idx == nullptr || q_w == nullptr || bank == nullptr || y == nullptr) return SDM_ERR_ARG;
    if (!checks::aligned16(bank) || !checks::aligned16(y)) return SDM_ERR_ALIGN;
    if (step_begin == step_end) return SDM_OK;
    ReadArgs a;
    memset(&a, 0, sizeof(a));
    a.q_idx = q_idx;
    a.q_w = q_w;
    a.bank = bank;
    a.y = y;
    a.status = status;
    a.P = shape->P;
    a.C = shape->C;
    a.R = shape->R;
    a.hd = shape->hd;
    a.nsl = (shape->hd + 127) / 128;
    a.valid_last = shape->valid_last;
    a.S = shape->S;
    a.steps = shape->steps;
    a.c0 = step_begin * shape->P;
    a.units = (step_end - step_begin) * shape->P * shape->C * a.nsl;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool wbf = shape->val_dtype == SDM_BF16;
    cudaError_t e;
    if (shape->bank_dtype == SDM_BF16)
        e = wbf ? launch_r<__nv_bfloat16, __nv_bfloat16>(a, cs) : launch_r<__nv_bfloat16, float>(a, cs);
    else
        e = wbf ? launch_r<float, __nv_bfloat16>(a, cs) : launch_r<float, float>(a, cs);
    return e == cudaSuccess ? SDM_OK : SDM_ERR_CUDA;
}
