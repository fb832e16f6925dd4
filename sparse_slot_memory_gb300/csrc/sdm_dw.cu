// sdm_dw.cu -- Phase-2 decay-and-write (DW) of the chunked sparse-delta-memory forward.
//
// Arithmetic (sparse-delta-memory 2.0.0, mover_da2_cuda.py and mover_fx_cuda.py module
// docstrings): per slot group of a chunk, in Phase-1 sorted order,
//   acc = 0; acc = fmaf(sc_m, dv[tok_m], acc) over the group's write entries;
//   bank[slot] = RN(fmaf(base, cpe_last, acc)), base = the row before this step,
// sc = k * expf(rex) and cpe_last (the value-type cpe widened) come from the Phase-1 record.
// A float32 bank stores the fmaf result itself. Every group is summed by one warp in sorted
// order and its row has one writer per step, so the result does not depend on the tiling.
//
// GB300 design: ONE persistent launch runs every step. Work items are (stream p, step, tile,
// 128-column slice); each stream has its own claim counter, items are claimed in (step, tile,
// slice) order, and an item of step t waits (bounded) until stream p's per-stream done counter
// shows every item of step t-1 finished. Claims are in order, so every item a warp waits on is
// already held by a running warp: no co-residency is needed and nothing can deadlock. While it
// waits, a warp prefetches its groups' bank rows into L2 (cp.async.bulk.prefetch), so the next
// step's random row reads are L2 hits by the time its predecessor finishes. Rows move as 8-byte
// (bf16) / 16-byte (f32) lane vectors, 256 / 512 bytes per warp access; records are staged per
// warp in shared memory; per 8-entry sub-batch every token-row and base-row load is issued
// before the dependent FMAs.
#include <cuda_bf16.h>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kDwThreads = 256;
constexpr int kDwWarps = kDwThreads / 32;

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// A lane's 4 columns of a row, kept in the storage type until used: 8 bytes (bf16) / 16 bytes (f32).
template <typename T>
struct Raw4;
template <>
struct Raw4<float> {
    float4 v;
    __device__ __forceinline__ void zero() { v = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void ld_nc(const float* p) { v = __ldg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ void ld_cg(const float* p) { v = __ldcg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ float operator[](int i) const { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
};
template <>
struct Raw4<__nv_bfloat16> {
    uint2 v;
    __device__ __forceinline__ void zero() { v = make_uint2(0u, 0u); }
    __device__ __forceinline__ void ld_nc(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint2*>(p)); }
    __device__ __forceinline__ void ld_cg(const __nv_bfloat16* p) { v = __ldcg(reinterpret_cast<const uint2*>(p)); }
    __device__ __forceinline__ float operator[](int i) const {
        const uint32_t w = i < 2 ? v.x : v.y;
        return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};

__device__ __forceinline__ void st4(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float (&o)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(o[2], o[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// Waits until *ctr >= need (lane 0 of the warp). Bounded: gives up after timeout_ns or when
// another warp raised the abort flag; on a timeout sets the status bit and the abort flag.
__device__ bool wait_done(const DWArgs& a, const uint32_t* ctr, uint32_t need) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        if (ld_acquire(ctr) < need) {
            const unsigned long long t0 = globaltimer();
            unsigned ns = 32;
            for (uint32_t it = 0;; ++it) {
                if (ld_acquire(ctr) >= need) break;
                if (ld_relaxed(a.abort_flag) != 0u) {
                    ok = false;
                    break;
                }
                if (globaltimer() - t0 > a.timeout_ns || it > (1u << 28)) {
                    atomicOr(a.status, kDevTimeout);
                    atomicExch(a.abort_flag, 1u);
                    ok = false;
                    break;
                }
                __nanosleep(ns);
                ns = ns < 512 ? ns * 2 : 512;
            }
        }
    }
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

template <typename BankT, typename DvT>
__global__ void __launch_bounds__(kDwThreads, 4) dw_kernel(const DWArgs a) {
    __shared__ int4 recs_s[kDwWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int4* const rs = recs_s[warp];
    BankT* const bank = static_cast<BankT*>(a.bank);
    const DvT* const dv = static_cast<const DvT*>(a.dv);
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kDwWarps + warp;
    int p = static_cast<int>(gwarp % a.P);
    int exhausted = 0;
    while (exhausted < a.P) {
        if (ld_relaxed(a.abort_flag) != 0u) return;
        uint32_t it = 0;
        if (lane == 0) it = atomicAdd(a.claim + p, 1u);
        it = __shfl_sync(kFull, it, 0);
        if (static_cast<int64_t>(it) >= a.per_stream) {
            p = p + 1 == a.P ? 0 : p + 1;
            ++exhausted;
            continue;
        }
        exhausted = 0;
        const int64_t ts = static_cast<int64_t>(it) / a.per_step;
        const int64_t rem = static_cast<int64_t>(it) - ts * a.per_step;
        const int tile = static_cast<int>(rem / a.nsl);
        const int sl = static_cast<int>(rem - static_cast<int64_t>(tile) * a.nsl);
        const int64_t ti = a.step_begin + ts;
        const int64_t c = ti * a.P + p;
        const int s0 = __ldg(a.tb + c * (a.ntk + 1) + tile);
        const int s1 = __ldg(a.tb + c * (a.ntk + 1) + tile + 1);
        const int col = sl * 128 + lane * 4;
        const bool active = col < a.hd;
        const int4* const rec = a.krec + c * a.nk;
        const int64_t brow0 = static_cast<int64_t>(p) * a.S;
        const int64_t drow0 = c * a.C;
        const uint32_t need = static_cast<uint32_t>(ts * a.per_step);

        if (ts > 0) {
            // Every item of a step > 0 waits, even an empty one: an item completes only after every
            // item of the earlier steps, so done >= t * per_step means steps < t are finished.
            // Before waiting: pull this item's first base rows into L2.
            if (s0 < s1 && ld_relaxed(a.done + p) < need) {
                const int m = s0 + lane;
                if (m < s1) {
                    const int4 r = __ldg(rec + m);
                    const uint32_t w0 = static_cast<uint32_t>(r.x);
                    if ((w0 & kLast) && !(w0 & kRecInvalid)) {
                        const int64_t row = brow0 + static_cast<uint32_t>(r.y);
                        const int w = min(128, a.hd - sl * 128);
                        const uint32_t bytes = static_cast<uint32_t>(w * sizeof(BankT));
                        const BankT* const src = bank + row * a.hd + sl * 128;
                        if (((bytes | static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src))) & 15u) == 0u)
                            prefetch_l2(src, bytes);
                    }
                }
            }
            if (!wait_done(a, a.done + p, need)) return;
        }

        constexpr int kSub = (sizeof(BankT) == 2 && sizeof(DvT) == 2) ? 8 : 4;   // entries per sub-batch
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int b = s0; b < s1; b += 32) {
            const int cnt = min(32, s1 - b);
            __syncwarp();
            if (lane < cnt) rs[lane] = __ldg(rec + b + lane);
            __syncwarp();
            for (int m = 0; m < cnt; m += kSub) {
                Raw4<DvT> dvv[kSub];
                Raw4<BankT> bv[kSub];
                // issue every token-row and base-row load of the sub-batch first
#pragma unroll
                for (int k = 0; k < kSub; ++k) {
                    const int4 r = rs[min(m + k, cnt - 1)];
                    const uint32_t w0 = static_cast<uint32_t>(r.x);
                    const bool in = m + k < cnt && active;
                    dvv[k].zero();
                    bv[k].zero();
                    if (in && !(w0 & kRecInvalid)) dvv[k].ld_nc(dv + (drow0 + (w0 & kRecTokMask)) * a.hd + col);
                    if (in && (w0 & kLast) && !(w0 & kRecInvalid))
                        bv[k].ld_cg(bank + (brow0 + static_cast<uint32_t>(r.y)) * a.hd + col);
                }
#pragma unroll
                for (int k = 0; k < kSub; ++k) {
                    if (m + k < cnt) {
                        const int4 r = rs[m + k];
                        const uint32_t w0 = static_cast<uint32_t>(r.x);
                        const float sc = __int_as_float(r.z);
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[i] = fmaf(sc, dvv[k][i], acc[i]);
                        if (w0 & kLast) {
                            if (!(w0 & kRecInvalid) && active) {
                                const float cp = __int_as_float(r.w);
                                float o[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[i] = fmaf(bv[k][i], cp, acc[i]);
                                st4(bank + (brow0 + static_cast<uint32_t>(r.y)) * a.hd + col, o);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc[i] = 0.f;
                        }
                    }
                }
            }
        }
        // publish: every lane's row stores before the stream's done count
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_add(a.done + p, 1u);
    }
}

template <typename BankT, typename DvT>
cudaError_t launch_t(const DWArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dw_kernel<BankT, DvT>, kDwThreads, 0);
    if (e != cudaSuccess) return e;
    per_sm = per_sm < 1 ? 1 : per_sm;
    const int64_t items = a.per_stream * a.P;
    int64_t blocks = static_cast<int64_t>(sms) * per_sm;
    const int64_t need_blocks = (items + kDwWarps - 1) / kDwWarps;
    if (blocks > need_blocks) blocks = need_blocks;
    if (blocks < 1) blocks = 1;
    dw_kernel<BankT, DvT><<<static_cast<unsigned>(blocks), kDwThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dw(const DWArgs& a, int dv_bf16, int bank_bf16, cudaStream_t stream) {
    if (a.per_stream <= 0) return cudaSuccess;
    if (bank_bf16) {
        return dv_bf16 ? launch_t<__nv_bfloat16, __nv_bfloat16>(a, stream) : launch_t<__nv_bfloat16, float>(a, stream);
    }
    return dv_bf16 ? launch_t<float, __nv_bfloat16>(a, stream) : launch_t<float, float>(a, stream);
}

}  // namespace sdm
