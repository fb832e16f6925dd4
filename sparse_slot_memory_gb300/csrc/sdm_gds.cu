// sdm_gds.cu -- GDS, the read side of the chunked sparse-delta-memory backward, one step at a
// time, and its C entry point sdm_gds (include/sdm.h).
//
// Arithmetic (sparse-delta-memory 2.0.0, mover_da2_cuda.py: module docstring, the "GDS, split by
// data need" comment and its read-records kernel), per chunk c = ti * P + p of the step:
//   (1) dots in token order: d_q_w[c, t, r] = <gr[c, t], bank[p*S + q_idx[c, t, r]]> for the valid
//       tokens t (0 for padding tokens);
//   (2) the grad scatter in sorted order: per read group (slot s, members m in Phase-1 sorted order)
//       acc = 0; acc = fmaf(sc_m, gr[c, tok_m], acc); grad[p*S + s] = RN(grad[p*S + s] + acc),
//       sc = f32(q) * expf(log_q) (the read record's scale).
// A dot is summed like every dot of the backward here: per lane an fmaf chain over its 4 columns of a
// 128-column slice, the 32 lane partials in one fixed lane tree (rows::allsum / rows::tsum16), the
// slices added in order from 0.
//
// GB300 design: two launches per step. The dots: one warp per token, the bank rows of 16 read
// entries in flight at once, their 16 dots reduced across the lanes together (transposed), lane e
// storing entry e. The scatter: a CTA of 8 warps per (chunk, tile of 256 sorted read positions), a
// warp the groups whose FIRST lies in its 32 positions; all lanes load their entries' scalars at
// once; the groups that end inside the warp's positions stream the token rows and their grad rows
// through a per-warp cp.async ring 8 positions deep (each lane copies and reads back its own 4
// columns); a group that runs past them (a hot slot) is walked afterwards in windows of 32 members.
// Every grad row is written by one warp once per launch (a single writer: no atomics).
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "sdm_checks.cuh"
#include "sdm_internal.cuh"
#include "sdm_rows.cuh"

namespace sdm {
namespace {

using namespace rows;

constexpr int kGdsThreads = 256;
constexpr int kGdsWarps = kGdsThreads / 32;
constexpr int kGdsTile = kGdsThreads;      // sorted read positions per scatter CTA: 32 per warp
constexpr int kGdsRing = 8;                // in-window positions whose rows are in flight (per warp)
constexpr uint32_t kGdsSentinel = kFirst | kLast | kInvalidBit;

struct GDSArgs {
    const int32_t* sorted_q;   // [N, nq]
    const int32_t* q_idx;      // [N, C, R]
    const void* q_val;         // [N, C, R] value type
    const float* log_q;        // [N, C, R]
    const float* gr;           // [N, C, hd]
    const void* bank;          // [P * S, hd] bank type
    void* grad;                // [P * S, hd] grad type
    float* d_q_w;              // [N, C, R]
    uint32_t* status;          // nullable
    int P, C, R, nq, hd, nsl, tiles, dgroups;
    int valid;                 // valid tokens of this step's chunks
    int64_t S, c0;             // c0: the step's first chunk
};

__device__ __forceinline__ bool valid_first(uint32_t v) { return (v & kFirst) != 0 && (v & kInvalidBit) == 0; }

// ---- (1) dots, one warp per token -----------------------------------------------------------------
template <typename BankT>
__global__ void __launch_bounds__(kGdsThreads) gds_dots_kernel(const GDSArgs a) {
    // launched as a programmatic dependent of the kernel before it (the previous step's kernel, or any
    // kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cl = static_cast<int>(blockIdx.x / a.dgroups);
    const int dg = static_cast<int>(blockIdx.x - static_cast<int64_t>(cl) * a.dgroups);
    const int t = dg * kGdsWarps + warp;
    if (t >= a.C) return;   // warp-uniform
    const int64_t c = a.c0 + cl;
    const int hd = a.hd, R = a.R;
    const bool tvalid = t < a.valid;
    const BankT* const bank = static_cast<const BankT*>(a.bank) + static_cast<int64_t>(cl) * a.S * hd;
    const float* const grow = a.gr + (c * a.C + t) * static_cast<int64_t>(hd);
    const int32_t* const qi = a.q_idx + (c * a.C + t) * static_cast<int64_t>(R);
    float* const drow = a.d_q_w + (c * a.C + t) * static_cast<int64_t>(R);
    uint32_t bad = 0;
    for (int e0 = 0; e0 < R; e0 += 16) {
        // lane e < 16 holds the slot of entry e0 + e (-1: no row)
        int32_t myslot = -1;
        if (tvalid && lane < 16 && e0 + lane < R) {
            myslot = __ldg(qi + e0 + lane);
            if (myslot < 0 || static_cast<int64_t>(myslot) >= a.S) {
                myslot = -1;
                bad = 1u;
            }
        }
        float total = 0.f;   // lane l: entry e0 + (l & 15)
        for (int sl = 0; sl < a.nsl; ++sl) {
            const int col = sl * 128 + lane * 4;
            const bool on = col < hd;
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            if (on && tvalid) ld4(grow + col, x);
            // the 16 entries' bank rows, all in flight: every load is unconditional (a lane without a
            // row reads row 0 / column 0 of the stream and drops the value), so none waits on a branch
            const uint32_t hasrow = __ballot_sync(kFull, myslot >= 0);
            const int ccol = on ? col : 0;
            Raw4<BankT> m[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int32_t s = __shfl_sync(kFull, myslot, e);
                m[e].ld(bank + static_cast<int64_t>(s < 0 ? 0 : s) * hd + ccol);
            }
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float mf[4];
                m[e].get(mf);
                const bool use = ((hasrow >> e) & 1u) && on;
#pragma unroll
                for (int i = 0; i < 4; ++i) mf[i] = use ? mf[i] : 0.f;
                v[e] = dot4(x, mf);
            }
            total += tsum16(v, lane);
        }
        if (lane < 16 && e0 + lane < R) drow[e0 + lane] = tvalid ? total : 0.f;
    }
    if (__any_sync(kFull, bad != 0) && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

// Rows of at most 128 columns and at most 16 read lanes (one slice, one block of entries): the same
// arithmetic as gds_dots_kernel, with a grid of resident warps only, each looping over tokens; the
// next token's ids and reading gradient load while the current token's bank rows are in flight.
template <typename BankT>
__global__ void __launch_bounds__(kGdsThreads) gds_dots_loop_kernel(const GDSArgs a, int total_warps) {
    // launched as a programmatic dependent of the kernel before it (the previous step's kernel, or any
    // kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int ntok = a.P * a.C;
    int it = blockIdx.x * kGdsWarps + (threadIdx.x >> 5);
    if (it >= ntok) return;   // warp-uniform
    const int hd = a.hd, R = a.R;
    const int col = lane * 4;
    const bool on = col < hd;
    const int ccol = on ? col : 0;
    uint32_t bad = 0;
    auto fetch = [&](int i, int32_t& slot, float (&x)[4]) {
        const int cl = i / a.C, t = i - cl * a.C;
        const int64_t tok = (a.c0 + cl) * a.C + t;
        slot = -1;
        x[0] = x[1] = x[2] = x[3] = 0.f;
        if (t < a.valid) {
            if (lane < R) {
                slot = __ldg(a.q_idx + tok * R + lane);
                if (slot < 0 || static_cast<int64_t>(slot) >= a.S) {
                    slot = -1;
                    bad = 1u;
                }
            }
            if (on) ld4(a.gr + tok * hd + col, x);
        }
    };
    int32_t myslot;
    float x[4];
    fetch(it, myslot, x);
    for (;;) {
        const int cl = it / a.C, t = it - cl * a.C;
        const int64_t tok = (a.c0 + cl) * a.C + t;
        const BankT* const bank = static_cast<const BankT*>(a.bank) + static_cast<int64_t>(cl) * a.S * hd;
        const uint32_t hasrow = __ballot_sync(kFull, myslot >= 0);
        Raw4<BankT> m[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int32_t s = __shfl_sync(kFull, myslot, e);
            m[e].ld(bank + static_cast<int64_t>(s < 0 ? 0 : s) * hd + ccol);
        }
        const int nit = it + total_warps;
        int32_t nslot = -1;
        float nx[4] = {0.f, 0.f, 0.f, 0.f};
        if (nit < ntok) fetch(nit, nslot, nx);
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            float mf[4];
            m[e].get(mf);
            const bool use = ((hasrow >> e) & 1u) && on;
#pragma unroll
            for (int i = 0; i < 4; ++i) mf[i] = use ? mf[i] : 0.f;
            v[e] = dot4(x, mf);
        }
        const float total = 0.f + tsum16(v, lane);
        if (lane < R) a.d_q_w[tok * R + lane] = t < a.valid ? total : 0.f;
        if (nit >= ntok) break;
        it = nit;
        myslot = nslot;
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = nx[i];
    }
    if (__any_sync(kFull, bad != 0) && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

// ---- (2) the grad scatter -------------------------------------------------------------------------
// One window of up to 32 members of a read group, lane i holding member i.
struct QMember {
    int n;          // members in this window
    bool last;      // the window holds the group's LAST
    bool ok;        // lane < n and the entry names a token and lane of the chunk
    int tok;
    float sc;
};

template <typename ValT>
__device__ __forceinline__ QMember qmember_window(const GDSArgs& a, const int32_t* srow, int q, int64_t c, int lane,
                                                  int32_t* slot_out) {
    QMember m;
    const int pos = q + lane;
    const uint32_t v = pos < a.nq ? static_cast<uint32_t>(__ldg(srow + pos)) : kGdsSentinel;
    const uint32_t lastm = __ballot_sync(kFull, (v & kLast) != 0);
    m.last = lastm != 0;
    m.n = m.last ? __ffs(lastm) : 32;
    const int t = static_cast<int>((v >> kTokenShift) & 0xFFu);
    const int r = static_cast<int>(v & 0xFFu);
    m.ok = lane < m.n && (v & kInvalidBit) == 0 && t < a.C && r < a.R;
    m.tok = m.ok ? t : 0;
    m.sc = 0.f;
    *slot_out = -1;
    if (m.ok) {
        const int64_t o = (c * a.C + t) * static_cast<int64_t>(a.R) + r;
        *slot_out = __ldg(a.q_idx + o);
        m.sc = widen(static_cast<const ValT*>(a.q_val)[o]) * expf(__ldg(a.log_q + o));
    }
    return m;
}

// A read group that starts at sorted position f and ends past its warp's 32 positions (a hot slot):
// windows of 32 members follow it to its LAST, the next window's scalars in flight while this one's
// rows arrive. Per block of 16 members the token rows are cp.async-copied into the warp's idle ring
// at once (each lane copies and reads back its own 4 columns, zeros past the row), then added in
// member order: the same fmaf chain as the in-window groups. No per-member branch: a member past the
// window or naming no entry of the chunk gets a zero-filled slot and has sc = 0, so it adds 0 (the
// walk runs on one warp and is bound by its dependency path: this made the skewed GDS 12 % faster).
template <typename GradT, typename ValT>
__device__ __noinline__ void open_read_group(const GDSArgs& a, const int32_t* srow, int64_t c, int cl, int f, int lane,
                                             uint32_t* bad, float4* buf) {
    GradT* const grad = static_cast<GradT*>(a.grad);
    const int hd = a.hd;
    const float* const gr_chunk = a.gr + c * a.C * static_cast<int64_t>(hd);
    int32_t s0;
    const QMember m0 = qmember_window<ValT>(a, srow, f, c, lane, &s0);
    (void)m0;
    const int32_t s = __shfl_sync(kFull, s0, 0);
    if (s < 0 || static_cast<int64_t>(s) >= a.S) {
        *bad = 1u;
        return;
    }
    const int64_t row = (static_cast<int64_t>(cl) * a.S + s) * hd;
    for (int sl = 0; sl < a.nsl; ++sl) {
        const int col = sl * 128 + lane * 4;
        const bool on = col < hd;
        const float* const gr_col = gr_chunk + (on ? col : 0);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        int32_t unused;
        QMember m = qmember_window<ValT>(a, srow, f, c, lane, &unused);
        for (int q = f;; q += 32) {
            QMember nm = m;
            if (!m.last) nm = qmember_window<ValT>(a, srow, q + 32, c, lane, &unused);
            const uint32_t okm = __ballot_sync(kFull, m.ok);
            for (int k0 = 0; k0 < m.n; k0 += 16) {   // k0 = 0 or 16
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int k = k0 + u;
                    const int tk = __shfl_sync(kFull, m.tok, k & 31);
                    const bool live = k < m.n && ((okm >> (k & 31)) & 1u);   // else the slot gets zeros
                    cp4z(reinterpret_cast<float*>(&buf[u * 32 + lane]), gr_col + static_cast<int64_t>(live ? tk : 0) * hd,
                         on && live);
                }
                cp_commit();
                cp_wait<0>();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int k = k0 + u;
                    const float scu = __shfl_sync(kFull, m.sc, k & 31);   // 0 past the window or naming no entry
                    float d[4];
                    get4(reinterpret_cast<const float*>(&buf[u * 32 + lane]), d);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(scu, d[i], acc[i]);
                }
            }
            if (m.last) break;
            m = nm;
        }
        if (on) {
            float g[4], o[4];
            ld4cg(grad + row + col, g);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = g[i] + acc[i];
            st4(grad + row + col, o);
        }
    }
}

// Shared memory of one scatter warp: a ring of positions, per position and lane the lane's 4 columns
// of the token's reading gradient (f32) and of the group's grad row.
template <typename GradT>
struct GdsRing {
    float4 gr[kGdsRing][32];
    GradT grad[kGdsRing][32][4];
    // a hot read group's walk reuses the ring as 16 token-row slots per lane
    float4 pad[sizeof(GradT) == 4 ? 0 : 16 - kGdsRing - kGdsRing / 2][32];
};

template <typename GradT, typename ValT>
__global__ void __launch_bounds__(kGdsThreads, 2) gds_scatter_kernel(const GDSArgs a) {
    // launched as a programmatic dependent of the kernel before it (the previous step's kernel, or any
    // kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ __align__(16) unsigned char gds_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    GdsRing<GradT>& ring = reinterpret_cast<GdsRing<GradT>*>(gds_smem)[warp];
    const int cl = static_cast<int>(blockIdx.x / a.tiles);
    const int tile = static_cast<int>(blockIdx.x - static_cast<int64_t>(cl) * a.tiles);
    const int64_t c = a.c0 + cl;
    const int nq = a.nq, hd = a.hd;
    const int32_t* const srow = a.sorted_q + c * nq;
    const int q0 = tile * kGdsTile + warp * 32;

    // this lane's sorted position and its entry's scalars (all lanes at once)
    const int pos = q0 + lane;
    const uint32_t v = pos < nq ? static_cast<uint32_t>(__ldg(srow + pos)) : kGdsSentinel;
    const int t = static_cast<int>((v >> kTokenShift) & 0xFFu), r = static_cast<int>(v & 0xFFu);
    const bool ok = (v & kInvalidBit) == 0 && t < a.C && r < a.R;
    int32_t slot = -1;
    float sc = 0.f;
    if (ok) {
        const int64_t o = (c * a.C + t) * static_cast<int64_t>(a.R) + r;
        slot = __ldg(a.q_idx + o);
        sc = widen(static_cast<const ValT*>(a.q_val)[o]) * expf(__ldg(a.log_q + o));
    }
    const uint32_t fmask = __ballot_sync(kFull, valid_first(v));
    const uint32_t lmask = __ballot_sync(kFull, ok && (v & kLast) != 0);
    const uint32_t okmask = __ballot_sync(kFull, ok);
    if (fmask == 0) return;   // no group starts here

    const int f0 = __ffs(fmask) - 1;
    const int flast = 31 - __clz(fmask);
    const bool open = (lmask >> flast) == 0u;
    const int cend = open ? flast - 1 : 31 - __clz(lmask);
    GradT* const grad_s = static_cast<GradT*>(a.grad) + static_cast<int64_t>(cl) * a.S * hd;   // the stream's rows
    const float* const gr_chunk = a.gr + c * a.C * static_cast<int64_t>(hd);
    uint32_t bad = 0;
    if (cend >= f0) {
        for (int sl = 0; sl < a.nsl; ++sl) {
            const int col = sl * 128 + lane * 4;
            const bool on = col < hd;
            const int ccol = on ? col : 0;   // a lane past the row copies nothing (zero fill) from column 0
            // position k's rows go to ring slot (k - f0) % kGdsRing: its token's reading gradient and,
            // for a group's FIRST, the group's grad row; one commit group per position
            auto issue = [&](int k) {
                if (k <= cend) {   // warp-uniform
                    const int ks = (k - f0) & (kGdsRing - 1);
                    const int tk = __shfl_sync(kFull, t, k);
                    const int32_t sk = __shfl_sync(kFull, slot, k);
                    if ((okmask >> k) & 1u)
                        cp4z(reinterpret_cast<float*>(&ring.gr[ks][lane]), gr_chunk + tk * hd + ccol, on);
                    if (((fmask >> k) & 1u) && sk >= 0 && static_cast<int64_t>(sk) < a.S)
                        cp4z(&ring.grad[ks][lane][0], grad_s + static_cast<int64_t>(sk) * hd + ccol, on);
                }
                cp_commit();
            };
#pragma unroll 1
            for (int k = f0; k < f0 + kGdsRing - 1; ++k) issue(k);
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, cg[4] = {0.f, 0.f, 0.f, 0.f};
            int64_t crow = 0;
            bool cbad = true;
#pragma unroll 4
            for (int k = f0; k <= cend; ++k) {
                issue(k + kGdsRing - 1);
                cp_wait<kGdsRing - 1>();   // position k's copies have landed (zeros past the row)
                const int ks = (k - f0) & (kGdsRing - 1);
                if ((fmask >> k) & 1u) {   // a group starts
                    const int32_t sk = __shfl_sync(kFull, slot, k);
                    cbad = sk < 0 || static_cast<int64_t>(sk) >= a.S;
                    crow = static_cast<int64_t>(cbad ? 0 : sk) * hd + ccol;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = 0.f;
                    if (cbad) bad = 1u;
                    else get4(&ring.grad[ks][lane][0], cg);
                }
                const float skk = __shfl_sync(kFull, sc, k);
                if (!cbad && ((okmask >> k) & 1u)) {
                    float d[4];
                    get4(reinterpret_cast<const float*>(&ring.gr[ks][lane]), d);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(skk, d[i], acc[i]);
                }
                if (((lmask >> k) & 1u) && !cbad && on) {   // the group ends: one rounding per element
                    float o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = cg[i] + acc[i];
                    st4(grad_s + crow, o);
                }
            }
            cp_wait<0>();
        }
    }
    static_assert(sizeof(GdsRing<GradT>) >= 16 * 32 * sizeof(float4), "the ring holds 16 rows per lane");
    if (open) open_read_group<GradT, ValT>(a, srow, c, cl, q0 + flast, lane, &bad, reinterpret_cast<float4*>(&ring));
    if (bad && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

template <typename GradT>
constexpr size_t gds_smem_bytes() { return sizeof(GdsRing<GradT>) * kGdsWarps; }

template <typename GradT, typename ValT>
cudaError_t launch_scatter(const GDSArgs& a, cudaStream_t stream) {
    constexpr size_t smem = gds_smem_bytes<GradT>();
    cudaError_t e = cudaFuncSetAttribute(gds_scatter_kernel<GradT, ValT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_dependent(gds_scatter_kernel<GradT, ValT>, dim3(static_cast<unsigned>(a.P) * a.tiles), dim3(kGdsThreads),
                            smem, stream, a);
}

template <typename BankT>
cudaError_t launch_dots(const GDSArgs& a, cudaStream_t stream) {
    if (a.nsl == 1 && a.R <= 16) {
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gds_dots_loop_kernel<BankT>, kGdsThreads, 0);
        if (e != cudaSuccess) return e;
        const int ntok = a.P * a.C;
        const int blocks = std::max(1, std::min((ntok + kGdsWarps - 1) / kGdsWarps, sms * std::max(per_sm, 1)));
        return launch_dependent(gds_dots_loop_kernel<BankT>, dim3(blocks), dim3(kGdsThreads), 0, stream, a,
                                blocks * kGdsWarps);
    }
    return launch_dependent(gds_dots_kernel<BankT>, dim3(static_cast<unsigned>(a.P) * a.dgroups), dim3(kGdsThreads), 0,
                            stream, a);
}

cudaError_t launch_gds(const GDSArgs& a, int grad_bf16, int bank_bf16, int val_bf16, cudaStream_t stream) {
    cudaError_t e = bank_bf16 ? launch_dots<__nv_bfloat16>(a, stream) : launch_dots<float>(a, stream);
    if (e != cudaSuccess) return e;
    if (grad_bf16)
        return val_bf16 ? launch_scatter<__nv_bfloat16, __nv_bfloat16>(a, stream)
                        : launch_scatter<__nv_bfloat16, float>(a, stream);
    return val_bf16 ? launch_scatter<float, __nv_bfloat16>(a, stream) : launch_scatter<float, float>(a, stream);
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" sdm_status sdm_gds(const sdm_shape* shape, int32_t grad_dtype, const int32_t* sorted_q,
                              const int32_t* q_idx, const void* q_val, const float* log_q, const float* gr,
                              const void* bank, void* grad, float* d_q_w, int64_t step_begin, int64_t step_end,
                              uint32_t* status, sdm_stream_t stream) {
    const void* const ptrs[] = {sorted_q, q_idx, q_val, log_q, gr, bank, grad, d_q_w};
    const sdm_status st = checks::check_backward(shape, grad_dtype, step_begin, step_end, ptrs);
    if (st != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    GDSArgs a;
    memset(&a, 0, sizeof(a));
    a.sorted_q = sorted_q;
    a.q_idx = q_idx;
    a.q_val = q_val;
    a.log_q = log_q;
    a.gr = gr;
    a.bank = bank;
    a.grad = grad;
    a.d_q_w = d_q_w;
    a.status = status;
    a.P = shape->P;
    a.C = shape->C;
    a.R = shape->R;
    a.nq = shape->C * shape->R;
    a.hd = shape->hd;
    a.nsl = (shape->hd + 127) / 128;
    a.tiles = (a.nq + kGdsTile - 1) / kGdsTile;
    a.dgroups = (shape->C + kGdsWarps - 1) / kGdsWarps;
    a.S = shape->S;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // the backward runs the steps last to first
    for (int64_t ti = step_end - 1; ti >= step_begin; --ti) {
        a.c0 = ti * a.P;
        a.valid = ti == shape->steps - 1 ? shape->valid_last : shape->C;
        if (launch_gds(a, grad_dtype == SDM_BF16, shape->bank_dtype == SDM_BF16, shape->val_dtype == SDM_BF16, cs) !=
            cudaSuccess)
            return SDM_ERR_CUDA;
    }
    return SDM_OK;
}
