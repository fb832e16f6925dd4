// sdm_dw.cu -- Phase-2 decay-and-write (DW) of the chunked sparse-delta-memory forward.
//
// Arithmetic (sparse-delta-memory 2.0.0, mover_da2_cuda.py and mover_fx_cuda.py module
// docstrings): per slot group of a chunk, in Phase-1 sorted order,
//   acc = 0; acc = fmaf(sc_m, dv[tok_m], acc) over the group's write entries;
//   bank[slot] = RN(fmaf(base, cpe_last, acc)), base = the row before this step,
// sc = k * expf(rex) and cpe_last (the value-type cpe widened) come from the Phase-1 record.
// A float32 bank stores the fmaf result itself. Steps apply in order.
//
// GB300 design: ONE launch runs every step, with no synchronization between warps. Each
// stream's slots fall into B buckets by a hash of the slot; a work item is (stream p, bucket b,
// 128-column slice) and one warp walks ALL steps of the item in order: step t of stream p
// touches bucket b through the contiguous record range [bb[t][b], bb[t][b+1]) of the chunk (Phase 1
// writes the records of each bucket's slot groups together). A bank row is written only by its
// bucket's warp, and a lane always handles the same 4 columns of every row, so a row rewritten
// in a later step is re-read by the very thread that stored it: program order alone orders the
// steps. Per group the arithmetic and order are those of a step-by-step DW, so the bits are
// the same. Items are claimed from one counter (load balance across uneven buckets).
// Rows move as 8-byte (bf16) / 16-byte (f32) lane vectors: 256 / 512 contiguous bytes per warp
// access. The item's records of up to 32 steps are taken as one sequence in step order, in
// windows of 32 that arrive in shared memory by cp.async two windows ahead; per sub-batch of up
// to 8 records every token-row and base-row load is issued before the dependent FMAs. A
// sub-batch never holds two records of one slot (those are of different steps): it is cut
// before the second, whose base row is then loaded after the first one's store. A long group
// (a hot slot's many write entries in one chunk) is one reference record here: its sum comes
// from long_kernel, which ran before over the group's own records in the same order.
#include <cuda_bf16.h>

#include <type_traits>
#include <utility>

#include "sdm_internal.cuh"
#include "sdm_rows.cuh"

namespace sdm {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kDwThreads = 224;   // 7 warps: 4 blocks (28 warps) per SM at <= 72 registers
constexpr int kDwWarps = kDwThreads / 32;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Long groups (at least kLongMin write entries in one chunk, e.g. the hot slots of a skewed
// stream): one warp per (group, 128-column slice) sums the group's tail records in order,
// acc = fmaf(sc_m, dv[tok_m], acc) from 0 -- the very chain of the DW walk -- with the token rows of
// 16 records in flight at a time. The DW walk meets the group as one reference record and takes the
// sum there, so a hot slot's terms no longer form one long chain inside its bucket's warp: all long
// groups of all steps are summed in parallel.
template <typename DvT>
__global__ void __launch_bounds__(kDwThreads) long_kernel(const LongArgs a) {
    // Launched as a programmatic dependent of the kernel before it (Phase 1): nothing is read or
    // written before that grid completes and its memory is visible. It does not trigger its own
    // dependent (the DW) early: DW blocks resident during Phase 1's last wave made the forward slower
    // (large workload 711 -> 753 us, wide_ragged 181 -> 198 us); the DW launches at this grid's end.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.claim = 0u;   // the DW's work counter (the DW waits for this grid)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const DvT* const dv = static_cast<const DvT*>(a.dv);
    const uint32_t hdu = static_cast<uint32_t>(a.hd);
    // a block per chunk, a grid of at most four blocks per SM looping over the chunks (on uniform
    // slots nothing is to be done: the kernel is only its launch)
    for (int64_t cb = blockIdx.x; cb < a.nchunks; cb += gridDim.x) {
        const int64_t c = a.c0 + cb;
        const int nl = a.lcnt[c];
        for (int item = warp; item < nl * a.nsl; item += kDwWarps) {
            const int li = item / a.nsl, sl = item - li * a.nsl;
            const int col = sl * 128 + lane * 4;
            const bool active = col < a.hd;
            const int4* const rec = a.krec + c * a.rstride;
            const DvT* const dv_lane = dv + static_cast<int64_t>(c) * a.C * a.hd + col;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            // records from the group's first tail record to its LAST (never past the chunk's records)
            for (int base = a.ldesc[c * a.maxL + li]; base < a.rstride; base += 16) {
                int4 r = make_int4(0, 0, 0, 0);
                const bool in = lane < 16 && base + lane < a.rstride;
                if (in) r = __ldcg(rec + base + lane);
                const uint32_t lastm = __ballot_sync(kFull, in && (static_cast<uint32_t>(r.x) & kLast));
                const int n = lastm ? __ffs(lastm) : 16;   // the group's records in this batch
                rows::Raw4<DvT> dvv[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint32_t w0 = __shfl_sync(kFull, static_cast<uint32_t>(r.x), k);
                    if (k < n && active && base + k < a.rstride) dvv[k].ld(dv_lane + static_cast<uint64_t>(w0 & kRecTokMask) * hdu);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float sc = __int_as_float(__shfl_sync(kFull, r.z, k));
                    if (k < n && base + k < a.rstride) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[i] = fmaf(sc, dvv[k][i], acc[i]);
                    }
                }
                if (lastm != 0u) break;
            }
            if (active)
                __stcg(reinterpret_cast<float4*>(a.lacc + (static_cast<int64_t>(c) * a.maxL + li) * a.hd + col),
                       make_float4(acc[0], acc[1], acc[2], acc[3]));
        }
    }
}

// the row's raw bytes (the dense snapshot is a copy of the base row)
__device__ __forceinline__ void raw_st(float* p, const rows::Raw4<float>& r) { *reinterpret_cast<float4*>(p) = r.v; }
__device__ __forceinline__ void raw_st(__nv_bfloat16* p, const rows::Raw4<__nv_bfloat16>& r) {
    *reinterpret_cast<uint2*>(p) = r.v;
}

// SNAP: the saving forward (a.snap is the dense compact snapshot)
template <typename BankT, typename DvT, bool SNAP>
__global__ void __launch_bounds__(kDwThreads, 4) dw_kernel(const DWArgs a) {
    // a programmatic dependent of the long-group kernel: nothing is touched before it completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int kSub = 8;   // entries per sub-batch (4 blocks of 7 warps per SM, 72 registers)
    // per warp three window buffers of 32 records (+ 8 slots read by the unrolled loads, never
    // used) and each record's first dv row (its chunk * C)
    __shared__ __align__(16) int4 recs_s[kDwWarps][3][40];
    __shared__ long long drow_s[kDwWarps][3][40];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    BankT* const bank = static_cast<BankT*>(a.bank);
    const DvT* const dv = static_cast<const DvT*>(a.dv);
    const int64_t nsteps = a.step_end - a.step_begin;
    const uint32_t hdu = static_cast<uint32_t>(a.hd);
    for (;;) {
        uint32_t it = 0;
        if (lane == 0) it = atomicAdd(a.claim, 1u);
        it = __shfl_sync(kFull, it, 0);
        if (static_cast<int64_t>(it) >= a.items) return;
        const int sl = static_cast<int>(it % static_cast<uint32_t>(a.nsl));
        const uint32_t rest = it / static_cast<uint32_t>(a.nsl);
        const int b = static_cast<int>(rest % static_cast<uint32_t>(a.B));
        const int p = static_cast<int>(rest / static_cast<uint32_t>(a.B));
        const int col = sl * 128 + lane * 4;
        const bool active = col < a.hd;
        BankT* const bank_lane = bank + static_cast<int64_t>(p) * a.S * a.hd + col;   // stream row 0, own columns
        const DvT* const dv_lane = dv + col;
        // bucket bounds [P][steps][B + 1]: step t's range of bucket b is [bb0[t * (B + 1)], bb0[t * (B + 1) + 1])
        const int32_t* const bb0 = a.bb + static_cast<int64_t>(p) * a.steps * (a.B + 1) + b;
        for (int64_t t0 = 0; t0 < nsteps; t0 += 32) {
            // The item's records of (up to) 32 steps, concatenated in step order: lane t holds
            // step t0 + t's range, cum the inclusive prefix of the counts.
            const int tn = static_cast<int>(nsteps - t0 < 32 ? nsteps - t0 : 32);
            int s0l = 0, cntl = 0;
            if (lane < tn) {
                const int32_t* const bt = bb0 + (a.step_begin + t0 + lane) * (a.B + 1);
                s0l = __ldg(bt);
                cntl = __ldg(bt + 1) - s0l;
            }
            int cum = cntl;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(kFull, cum, d);
                if (lane >= d) cum += y;
            }
            const int total = __shfl_sync(kFull, cum, 31);
            if (total == 0) continue;
            const int64_t cl = (a.step_begin + t0 + lane) * a.P + p;   // lane t's chunk
            const long long rbase = cl * a.rstride + s0l - (cum - cntl);   // record of position g: rbase + g
            const long long dbase = static_cast<long long>(cl) * a.C;
            const int nwin = (total + 31) >> 5;
            // window w (positions 32w..) into buffer s: lane j fetches position 32w + j by cp.async
            auto fetch = [&](int w, int s) {
                const int g = w * 32 + lane;
                int ts = 0;   // the step holding g: the number of steps whose inclusive count is <= g
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) {
                    const int c = __shfl_sync(kFull, cum, ts + d - 1);
                    if (c <= g) ts += d;
                }
                const long long rb = __shfl_sync(kFull, rbase, ts);
                const long long db = __shfl_sync(kFull, dbase, ts);
                if (g < total) {
                    cp_async16(&recs_s[warp][s][lane], a.krec + rb + g);
                    drow_s[warp][s][lane] = db;
                }
                cp_async_commit();
            };
            __syncwarp();
            fetch(0, 0);
            if (nwin > 1) fetch(1, 1);
            cp_async_wait_all();
            __syncwarp();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t gord = 0;   // the current group's dense ordinal (from its FIRST record)
            for (int w = 0; w < nwin; ++w) {
                const int s = w % 3;
                if (w + 2 < nwin) fetch(w + 2, (w + 2) % 3);
                const int n = min(32, total - w * 32);
                const int4* const rs = recs_s[warp][s];
                const long long* const ds = drow_s[warp][s];
                // A record whose slot is also the LAST slot of an earlier record of the window (an
                // earlier step) must load its base row after that record's store: prev = the
                // nearest such record.
                uint32_t key = 0x80000000u | static_cast<uint32_t>(lane);
                if (lane < n && (static_cast<uint32_t>(rs[lane].x) & kLast)) key = static_cast<uint32_t>(rs[lane].y);
                const uint32_t same = __match_any_sync(kFull, key) & lt;
                const int prev = same ? 31 - __clz(same) : -1;
                // One sub-batch of up to K records [m, m + cnt): every token-row and base-row load
                // first, then the FMA chain in order.
                auto sub = [&](int m, int cnt, auto kw) {
                    constexpr int K = decltype(kw)::value;
                    rows::Raw4<DvT> dvv[K];
                    rows::Raw4<BankT> bv[K];
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        const int4 r = rs[m + k];
                        const uint32_t w0 = static_cast<uint32_t>(r.x);
                        if (k < cnt && active) {
                            dvv[k].ld(dv_lane + static_cast<uint64_t>(ds[m + k] + (w0 & kRecTokMask)) * hdu);
                            if (w0 & kLast) bv[k].ld_cg(bank_lane + static_cast<uint64_t>(static_cast<uint32_t>(r.y)) * hdu);
                        }
                    }
                    asm volatile("" ::: "memory");   // the records are read again below, not held in registers
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        if (k < cnt) {
                            const int4 r = rs[m + k];
                            const uint32_t w0 = static_cast<uint32_t>(r.x);
                            const float sc = __int_as_float(r.z);
                            if (SNAP && (w0 & kFirst)) gord = (w0 >> kRecOrdShift) & kRecOrdMask;
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc[i] = fmaf(sc, dvv[k][i], acc[i]);
                            if (w0 & kLast) {
                                if (SNAP && active)   // saving forward: the base row, raw
                                    raw_st(static_cast<BankT*>(a.snap) +
                                               (static_cast<uint64_t>(ds[m + k]) * a.W + gord) * hdu + col,
                                           bv[k]);
                                if (active) {
                                    const float cp = __int_as_float(r.w);
                                    float o[4];
#pragma unroll
                                    for (int i = 0; i < 4; ++i) o[i] = fmaf(bv[k][i], cp, acc[i]);
                                    rows::st4cs(bank_lane + static_cast<uint64_t>(static_cast<uint32_t>(r.y)) * hdu, o);
                                }
#pragma unroll
                                for (int i = 0; i < 4; ++i) acc[i] = 0.f;
                            }
                        }
                    }
                };
                // A long group's reference record: base row, its precomputed sum, the row back (on its
                // own: sub-batches stop before it).
                auto long_ref = [&](int m) {
                    const int4 r = rs[m];
                    if (active) {
                        BankT* const row = bank_lane + static_cast<uint64_t>(static_cast<uint32_t>(r.y)) * hdu;
                        rows::Raw4<BankT> bv;
                        bv.ld_cg(row);
                        const float4 la = __ldcg(reinterpret_cast<const float4*>(
                            a.lacc + static_cast<uint64_t>(static_cast<uint32_t>(r.z)) * hdu + col));
                        if constexpr (SNAP)
                            raw_st(static_cast<BankT*>(a.snap) +
                                       (static_cast<uint64_t>(ds[m]) * a.W + ((static_cast<uint32_t>(r.x) >> kRecOrdShift) & kRecOrdMask)) * hdu + col,
                                   bv);
                        const float cp = __int_as_float(r.w);
                        const float o[4] = {fmaf(bv[0], cp, la.x), fmaf(bv[1], cp, la.y), fmaf(bv[2], cp, la.z),
                                            fmaf(bv[3], cp, la.w)};
                        rows::st4cs(row, o);
                    }
                };
                const uint32_t longm = __ballot_sync(kFull, lane < n && (static_cast<uint32_t>(rs[lane].x) & kRecLong));
                for (int m = 0; m < n;) {
                    if ((longm >> m) & 1u) {
                        long_ref(m);
                        ++m;
                        continue;
                    }
                    int e = min(m + kSub, n);
                    const uint32_t cut = __ballot_sync(kFull, lane > m && lane < e && (prev >= m || ((longm >> lane) & 1u)));
                    if (cut) e = __ffs(cut) - 1;
                    if (e - m > kSub / 2)
                        sub(m, e - m, std::integral_constant<int, kSub>());
                    else
                        sub(m, e - m, std::integral_constant<int, kSub / 2>());
                    m = e;
                }
                cp_async_wait_all();   // window w + 1 (and the one after it, if issued)
                __syncwarp();
            }
        }
    }
}

template <typename BankT, typename DvT, bool SNAP>
cudaError_t launch_t1(const DWArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dw_kernel<BankT, DvT, SNAP>, kDwThreads, 0);
    if (e != cudaSuccess) return e;
    per_sm = per_sm < 1 ? 1 : per_sm;
    int64_t blocks = static_cast<int64_t>(sms) * per_sm;
    const int64_t need_blocks = (a.items + kDwWarps - 1) / kDwWarps;
    if (blocks > need_blocks) blocks = need_blocks;
    if (blocks < 1) blocks = 1;
    return launch_dependent(dw_kernel<BankT, DvT, SNAP>, dim3(static_cast<unsigned>(blocks)), dim3(kDwThreads), 0, stream, a);
}

template <typename BankT, typename DvT>
cudaError_t launch_t(const DWArgs& a, cudaStream_t stream) {
    return a.snap != nullptr ? launch_t1<BankT, DvT, true>(a, stream) : launch_t1<BankT, DvT, false>(a, stream);
}

}  // namespace

cudaError_t launch_long(const LongArgs& a, int dv_bf16, cudaStream_t stream) {
    if (a.nchunks <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.nchunks < 4 * static_cast<int64_t>(sms) ? a.nchunks : 4 * static_cast<int64_t>(sms)));
    return dv_bf16 ? launch_dependent(long_kernel<__nv_bfloat16>, grid, dim3(kDwThreads), 0, stream, a)
                   : launch_dependent(long_kernel<float>, grid, dim3(kDwThreads), 0, stream, a);
}

cudaError_t launch_dw(const DWArgs& a, int dv_bf16, int bank_bf16, cudaStream_t stream) {
    if (a.items <= 0 || a.step_end <= a.step_begin) return cudaSuccess;
    if (bank_bf16) {
        return dv_bf16 ? launch_t<__nv_bfloat16, __nv_bfloat16>(a, stream) : launch_t<__nv_bfloat16, float>(a, stream);
    }
    return dv_bf16 ? launch_t<float, __nv_bfloat16>(a, stream) : launch_t<float, float>(a, stream);
}

}  // namespace sdm
