// sdm_pa.cu -- Phase A of the chunked sparse-delta-memory backward: the backward of DW, one step
// at a time, and its C entry point sdm_pa (include/sdm.h).
//
// Arithmetic (sparse-delta-memory 2.0.0, pa_dc_cuda.py module docstring, "PA per write group", and
// its records kernel): per valid write group of a chunk (slot s, members m in Phase-1 sorted order),
// with gdw = grad[s] before the step and snap = the group's row of the dense compact snapshot,
//   sc_m = -beta[tok_m] * (f32(k_m) * expf(log_k_m))
//   acc = 0; acc = fmaf(sc_m, d_dva[tok_m], acc) over the members in order
//   grad[s] = RN(fmaf(gdw, cpe_last, acc))          (f32: the fmaf result itself)
//   bank[s] = snap                                    (raw copy of the pre-write row)
//   grad_g[e] = cpe_e * <gdw, snap>,  d_k_eff[e] = -beta[tok_e] * <d_dva[tok_e], snap>.
// Every dot is summed the same way whatever the tiling: a lane sums its 4 columns of a 128-column
// slice in column order (an fmaf chain), the 32 lane partials meet in one fixed tree (pairs of lanes
// l, l ^ h for h = 1, 2, 4, 8, 16; both partners of a pair add the same two values, so the sum does
// not depend on which lane computes it), and the slices' sums add in slice order from 0.
//
// GB300 design: one launch per step; a CTA of 8 warps takes one chunk and a tile of 256 sorted
// positions, a warp its 32 positions. All 32 lanes load their entries' scalars (slot, k, log_k, cpe,
// beta) at once. The dense ordinal of a group (its snapshot row) is the count of valid FIRST flags
// before it in the sorted row: each CTA counts the positions before its tile once. The rows of the
// groups that start and end in the warp's positions (nearly all of them) stream through a per-warp
// shared-memory ring: every lane cp.async-copies its own 4 columns of a position's token row and, at
// a group's FIRST, of the group's grad and snapshot rows, 8 positions ahead, and reads back only what
// it copied. Per aligned block of 8 positions the 16 dot partials (8 entry dots, 8 group dots) are
// reduced across the lanes together, transposed (16 shuffles for 16 sums), each landing in the lane
// of its position. A group that starts in the warp's positions and runs past them (a hot slot) is
// walked afterwards in windows of 32 members; it keeps each member's dot sum in d_k_eff between
// slices (the member's own lane stores and re-reads it), with the same arithmetic.
#include <cuda_bf16.h>

#include <cstring>

#include "sdm_checks.cuh"
#include "sdm_internal.cuh"
#include "sdm_rows.cuh"

namespace sdm {
namespace {

using namespace rows;

constexpr int kPaThreads = 256;
constexpr int kPaWarps = kPaThreads / 32;
constexpr int kPaTile = kPaThreads;        // sorted positions per CTA: 32 per warp
constexpr int kPaRing = 8;                 // in-window positions whose rows are in flight (per warp)
constexpr int kPaCountUnroll = 16;         // sorted words per thread in flight while counting FIRSTs
constexpr uint32_t kPaSentinel = kFirst | kLast | kInvalidBit;

struct PAArgs {
    const int32_t* sorted_k;   // [N, nk]
    const int32_t* k_idx;      // [N, C, W]
    const void* k_val;         // [N, C, W] value type
    const float* log_k;        // [N, C, W]
    const void* cpe;           // [N, C, W] value type
    const float* beta;         // [N, C]
    const float* dva;          // [N, C, hd]
    void* grad;                // [P * S, hd] grad type
    void* bank;                // [P * S, hd] bank type
    const void* snap;          // this step's snapshot rows: [P, nk, hd] bank type
    float* d_k_eff;            // [N, C, W]
    float* grad_g;             // [N, C, W]
    uint32_t* status;          // nullable
    int P, C, W, nk, hd, nsl, tiles;
    int64_t S, c0;             // c0: the step's first chunk
};

// raw copy of a lane's 4 columns (the snapshot row is the bank row's bytes)
__device__ __forceinline__ void copy4(float* d, const float* s) {
    *reinterpret_cast<float4*>(d) = __ldg(reinterpret_cast<const float4*>(s));
}
__device__ __forceinline__ void copy4(__nv_bfloat16* d, const __nv_bfloat16* s) {
    *reinterpret_cast<uint2*>(d) = __ldg(reinterpret_cast<const uint2*>(s));
}

// raw copy of a lane's 4 columns from shared memory (the snapshot row's bytes)
__device__ __forceinline__ void copy_raw4(float* d, const float* s) {
    *reinterpret_cast<float4*>(d) = *reinterpret_cast<const float4*>(s);
}
__device__ __forceinline__ void copy_raw4(__nv_bfloat16* d, const __nv_bfloat16* s) {
    *reinterpret_cast<uint2*>(d) = *reinterpret_cast<const uint2*>(s);
}

__device__ __forceinline__ bool valid_first(uint32_t v) { return (v & kFirst) != 0 && (v & kInvalidBit) == 0; }

// One window of up to 32 members of a group, lane i holding member i.
struct Member {
    int n;          // members in this window
    bool last;      // the window holds the group's LAST
    bool ok;        // lane < n and the entry names a token and lane of the chunk
    int tok;        // token (0 when !ok)
    int64_t o;      // entry index of the chunk's [C, W] arrays (global)
    float sc, cp, beta;
};

template <typename ValT>
__device__ __forceinline__ Member member_window(const PAArgs& a, const int32_t* srow, int q, int64_t c, int lane) {
    Member m;
    const int pos = q + lane;
    const uint32_t v = pos < a.nk ? static_cast<uint32_t>(__ldg(srow + pos)) : kPaSentinel;
    const uint32_t lastm = __ballot_sync(kFull, (v & kLast) != 0);
    m.last = lastm != 0;
    m.n = m.last ? __ffs(lastm) : 32;
    const int t = static_cast<int>((v >> kTokenShift) & 0xFFu);
    const int j = static_cast<int>(v & 0xFFu);
    m.ok = lane < m.n && (v & kInvalidBit) == 0 && t < a.C && j < a.W;
    m.tok = m.ok ? t : 0;
    m.o = c * a.nk + (m.ok ? t * a.W + j : 0);
    m.sc = 0.f;
    m.cp = 1.f;
    m.beta = 0.f;
    if (m.ok) {
        const float kv = widen(static_cast<const ValT*>(a.k_val)[m.o]);
        const float lk = __ldg(a.log_k + m.o);
        m.cp = widen(static_cast<const ValT*>(a.cpe)[m.o]);
        m.beta = __ldg(a.beta + c * a.C + t);
        m.sc = -m.beta * (kv * expf(lk));
    }
    return m;
}

// The hot-group walk's token rows stream through the warp's buffer in sub-blocks of kWalkSub members:
// sub-block g of a slice's walk (window g / 4, its members kWalkSub * (g % 4) .. + kWalkSub - 1) is
// cp.async-copied into slots kWalkSub * (g % kWalkDepth) .. + kWalkSub - 1 of the buffer (each lane
// copies and reads back its own 4 columns, zeros past the row), and kWalkDepth sub-blocks are in flight
// at once, across window boundaries (the next window's scalars are loaded one window ahead).
constexpr int kWalkSub = 8;
constexpr int kWalkDepth = 3;
constexpr int kWalkRows = kWalkSub * kWalkDepth;   // row slots per lane

// sub-block g's copies: members of a window with n members, tokens tok (lane k holds member k), okm
// the members that name an entry of the chunk; every slot of the sub-block is written (zeros for
// the others)
__device__ __forceinline__ void walk_issue(int g, int n, int tok, uint32_t okm, const float* dva_col, bool dva_on,
                                           int hd, int lane, float4* buf) {
    const int slot = g % kWalkDepth;
#pragma unroll
    for (int u = 0; u < kWalkSub; ++u) {
        const int k = kWalkSub * (g & 3) + u;
        const int tk = __shfl_sync(kFull, tok, k);
        const bool live = k < n && ((okm >> k) & 1u);   // else the slot gets zeros
        cp4z(reinterpret_cast<float*>(&buf[(slot * kWalkSub + u) * 32 + lane]),
             dva_col + static_cast<int64_t>(live ? tk : 0) * hd, dva_on && live);
    }
    cp_commit();
}

// wait until at most `pend` copy groups issued after the one needed are still in flight
__device__ __forceinline__ void walk_wait(int pend) {
    if (pend >= 2)
        cp_wait<2>();
    else if (pend == 1)
        cp_wait<1>();
    else
        cp_wait<0>();
}

// sub-block g of window m: acc += its terms (member order); v[OFF + u] = member u's dot partial.
// No per-member branch: a member past the window or naming no entry of the chunk has sc = 0 and a
// zero-filled slot, so it adds 0 (its dot partial is never used); the 8 members' shuffles and
// shared loads then issue together (a hot group's walk runs on one warp, bound by its own
// dependency path: this made the skewed Phase A 27 % faster).
template <int OFF>
__device__ __forceinline__ void walk_sub(const Member& m, int g, const float (&sn)[4], float (&acc)[4], float (&v)[16],
                                         int lane, const float4* buf) {
    const int slot = g % kWalkDepth;
#pragma unroll
    for (int u = 0; u < kWalkSub; ++u) {
        const int k = kWalkSub * (g & 3) + u;
        const float scu = __shfl_sync(kFull, m.sc, k);   // 0 for a member past the window or naming no entry
        float d[4];
        get4(reinterpret_cast<const float*>(&buf[(slot * kWalkSub + u) * 32 + lane]), d);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(scu, d[i], acc[i]);
        v[OFF + u] = dot4(d, sn);
    }
}

// Window w of the walk (members m; nm the next window's when `more`): acc += the window's terms on
// this lane's 4 columns in member order; returns this lane's member's <dva, snap> sum over the slice
// (lanes >= m.n get 0). The dot partials of 16 members are reduced across the lanes together
// (rows::tsum16, the tree of rows::allsum): member k's sum lands in lane k. `issued` counts the
// slice's sub-blocks issued so far (0 at the slice's first window).
__device__ __forceinline__ float window_terms(const Member& m, const Member& nm, bool more, int w, int& issued,
                                              const float* dva_col, bool dva_on, int hd, const float (&sn)[4],
                                              float (&acc)[4], int lane, float4* buf) {
    static_assert(kWalkSub == 8 && kWalkDepth <= 5, "4 sub-blocks per window; at most one window ahead");
    float mine = 0.f;
    const uint32_t okm = __ballot_sync(kFull, m.ok);
    const int nsb = (m.n + kWalkSub - 1) / kWalkSub;                  // this window's sub-blocks (1..4)
    const int nsn = more ? (nm.n + kWalkSub - 1) / kWalkSub : 0;      // the next window's
    uint32_t okn = 0u;
    bool have_okn = false;
    auto top_up = [&](int g) {   // sub-blocks up to g + kWalkDepth - 1 in flight
        while (issued < g + kWalkDepth) {
            const int wi = issued >> 2, ji = issued & 3;
            if (wi == w) {
                if (ji >= nsb) break;
                walk_issue(issued, m.n, m.tok, okm, dva_col, dva_on, hd, lane, buf);
            } else {
                if (ji >= nsn) break;   // wi == w + 1
                if (!have_okn) {
                    okn = __ballot_sync(kFull, nm.ok);
                    have_okn = true;
                }
                walk_issue(issued, nm.n, nm.tok, okn, dva_col, dva_on, hd, lane, buf);
            }
            ++issued;
        }
    };
    const int g0 = 4 * w;
    for (int h = 0; 2 * h < nsb; ++h) {   // members 16h .. 16h + 15: sub-blocks 2h and 2h + 1
        float v[16];
        top_up(g0 + 2 * h);
        walk_wait(issued - 1 - (g0 + 2 * h));
        walk_sub<0>(m, g0 + 2 * h, sn, acc, v, lane, buf);
        if (2 * h + 1 < nsb) {
            top_up(g0 + 2 * h + 1);
            walk_wait(issued - 1 - (g0 + 2 * h + 1));
            walk_sub<kWalkSub>(m, g0 + 2 * h + 1, sn, acc, v, lane, buf);
        } else {
#pragma unroll
            for (int u = 0; u < kWalkSub; ++u) v[kWalkSub + u] = 0.f;
        }
        const float red = tsum16(v, lane);
        if ((lane >> 4) == h) mine = red;
    }
    return mine;
}

// A group that starts at sorted position f and ends past its warp's 32 positions (a hot slot):
// windows of 32 members follow it to its LAST; slices outside, windows inside, each member's dot
// sum kept in d_k_eff between slices. Same arithmetic and order as the in-window groups.
template <typename GradT, typename BankT, typename ValT>
__device__ __noinline__ void open_group(const PAArgs& a, const int32_t* srow, int64_t c, int cl, int f, int ord,
                                        int lane, uint32_t* bad, float4* buf) {
    GradT* const grad = static_cast<GradT*>(a.grad);
    BankT* const bank = static_cast<BankT*>(a.bank);
    const BankT* const snap = static_cast<const BankT*>(a.snap);
    const int hd = a.hd;
    const float* const dva_chunk = a.dva + c * a.C * static_cast<int64_t>(hd);
    const Member m0 = member_window<ValT>(a, srow, f, c, lane);
    const int32_t s = __shfl_sync(kFull, m0.ok ? __ldg(a.k_idx + m0.o) : -1, 0);
    if (s < 0 || static_cast<int64_t>(s) >= a.S) {   // not a row of the bank: the group is dropped
        *bad = 1u;
        for (int q = f;; q += 32) {
            const Member m = member_window<ValT>(a, srow, q, c, lane);
            if (m.ok) a.d_k_eff[m.o] = a.grad_g[m.o] = 0.f;
            if (m.last) break;
        }
        return;
    }
    const int64_t row = (static_cast<int64_t>(cl) * a.S + s) * hd;
    const int64_t srow_g = (static_cast<int64_t>(cl) * a.nk + ord) * hd;
    float gsum = 0.f;
    for (int sl = 0; sl < a.nsl; ++sl) {
        const int col = sl * 128 + lane * 4;
        const bool on = col < hd;
        float g4[4] = {0.f, 0.f, 0.f, 0.f}, s4[4] = {0.f, 0.f, 0.f, 0.f};
        if (on) {
            ld4cg(grad + row + col, g4);
            ld4(snap + srow_g + col, s4);
            copy4(bank + row + col, snap + srow_g + col);
        }
        gsum += allsum(dot4(g4, s4));
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float cpl = 1.f;
        Member m = member_window<ValT>(a, srow, f, c, lane);
        int issued = 0;   // the walk's sub-blocks issued (this slice)
        for (int q = f, w = 0;; q += 32, ++w) {
            Member nm = m;
            if (!m.last) nm = member_window<ValT>(a, srow, q + 32, c, lane);   // the next window's scalars in flight
            const float r = window_terms(m, nm, !m.last, w, issued, dva_chunk + (on ? col : 0), on, hd, s4, acc, lane, buf);
            if (m.ok) {
                if (a.nsl == 1) {   // one slice: the sums are final
                    a.d_k_eff[m.o] = -m.beta * (0.f + r);
                    a.grad_g[m.o] = m.cp * gsum;
                } else {
                    a.d_k_eff[m.o] = (sl == 0 ? 0.f : a.d_k_eff[m.o]) + r;
                }
            }
            if (m.last) {
                cpl = __shfl_sync(kFull, m.cp, m.n - 1);
                break;
            }
            m = nm;
        }
        if (on) {
            float o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = fmaf(g4[i], cpl, acc[i]);
            st4(grad + row + col, o);
        }
    }
    if (a.nsl == 1) return;
    for (int q = f;; q += 32) {
        const Member m = member_window<ValT>(a, srow, q, c, lane);
        if (m.ok) {
            a.d_k_eff[m.o] = -m.beta * a.d_k_eff[m.o];
            a.grad_g[m.o] = m.cp * gsum;
        }
        if (m.last) break;
    }
}

// Shared memory of one warp: a ring of kPaRing positions, per position and lane the lane's 4 columns
// of the token row (f32), of the grad row and of the snapshot row.
template <typename GradT, typename BankT>
struct PaRing {
    float4 dva[kPaRing][32];
    GradT grad[kPaRing][32][4];
    BankT snap[kPaRing][32][4];
};

// One warp's shared memory: the ring, or (a hot group's walk, once the ring is idle) kWalkRows token-row
// slots per lane.
template <typename GradT, typename BankT>
union PaWarpSmem {
    PaRing<GradT, BankT> ring;
    float4 walk[kWalkRows][32];
};

template <typename GradT, typename BankT>
constexpr size_t pa_smem_bytes() { return sizeof(PaWarpSmem<GradT, BankT>) * kPaWarps; }

template <typename GradT, typename BankT, typename ValT>
__global__ void __launch_bounds__(kPaThreads, 2) pa_kernel(const PAArgs a) {
    // launched as a programmatic dependent of the kernel before it (the previous step's kernel, or any
    // kernel of the caller's): nothing is read or written before that grid completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ int before_s[kPaWarps];   // valid FIRSTs before the tile, per warp's share of the count
    __shared__ int in_s[kPaWarps];       // valid FIRSTs in each warp's 32 positions
    extern __shared__ __align__(16) unsigned char pa_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    PaWarpSmem<GradT, BankT>& wsm = reinterpret_cast<PaWarpSmem<GradT, BankT>*>(pa_smem)[warp];
    PaRing<GradT, BankT>& ring = wsm.ring;
    const int cl = static_cast<int>(blockIdx.x / a.tiles);   // stream of the chunk
    const int tile = static_cast<int>(blockIdx.x - static_cast<int64_t>(cl) * a.tiles);
    const int64_t c = a.c0 + cl;
    const int nk = a.nk, hd = a.hd;
    const int32_t* const srow = a.sorted_k + c * nk;
    const int r0 = tile * kPaTile;

    // ---- this lane's sorted position and its entry's scalars (all lanes at once) ----------------
    const int q0 = r0 + warp * 32;
    const int pos = q0 + lane;
    const uint32_t v = pos < nk ? static_cast<uint32_t>(__ldg(srow + pos)) : kPaSentinel;
    const int t = static_cast<int>((v >> kTokenShift) & 0xFFu), j = static_cast<int>(v & 0xFFu);
    const bool named = t < a.C && j < a.W;              // names an entry of the chunk
    const bool ok = (v & kInvalidBit) == 0 && named;
    const int64_t o = c * nk + (named ? t * a.W + j : 0);
    int32_t slot = -1;
    float sc = 0.f, cp = 1.f, be = 0.f;
    if (ok) {
        slot = __ldg(a.k_idx + o);
        const float kv = widen(static_cast<const ValT*>(a.k_val)[o]);
        const float lk = __ldg(a.log_k + o);
        cp = widen(static_cast<const ValT*>(a.cpe)[o]);
        be = __ldg(a.beta + c * a.C + t);
        sc = -be * (kv * expf(lk));
    }
    const uint32_t fmask = __ballot_sync(kFull, valid_first(v));
    const uint32_t lmask = __ballot_sync(kFull, ok && (v & kLast) != 0);
    const uint32_t okmask = __ballot_sync(kFull, ok);

    // ---- dense ordinal of the window's first group: valid FIRSTs before it ----------------------
    // (the loads of a thread's words are issued together: a 4096-entry row is one round trip)
    int before = 0;
    for (int i0 = threadIdx.x; i0 < r0; i0 += kPaThreads * kPaCountUnroll) {
        uint32_t wv[kPaCountUnroll];
#pragma unroll
        for (int u = 0; u < kPaCountUnroll; ++u) {
            const int i = i0 + u * kPaThreads;
            wv[u] = i < r0 ? static_cast<uint32_t>(__ldg(srow + i)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kPaCountUnroll; ++u) before += valid_first(wv[u]);
    }
    before = __reduce_add_sync(kFull, before);
    if (lane == 0) {
        before_s[warp] = before;
        in_s[warp] = __popc(fmask);
    }
    __syncthreads();
    int ord0 = 0;
#pragma unroll
    for (int w = 0; w < kPaWarps; ++w) ord0 += before_s[w] + (w < warp ? in_s[w] : 0);

    // invalid entries of these positions: zero outputs
    if ((v & kInvalidBit) != 0 && pos < nk && named) a.d_k_eff[o] = a.grad_g[o] = 0.f;
    if (fmask == 0) return;   // no group starts here (a previous warp's group, or invalid entries)

    // ---- the groups that start and end in this window: positions [f0, cend] ----------------------
    // The last group to start here may run past the window ("open"); it is walked afterwards.
    const int f0 = __ffs(fmask) - 1;
    const int flast = 31 - __clz(fmask);
    const bool open = (lmask >> flast) == 0u;
    const int cend = open ? flast - 1 : 31 - __clz(lmask);
    // this lane's group: the nearest FIRST at or before it (its lane index), -1 if none
    const uint32_t upto = fmask & (lane == 31 ? kFull : ((2u << lane) - 1u));
    const int myf = upto ? 31 - __clz(upto) : -1;
    const bool mine = ok && myf >= 0 && lane <= cend;    // this lane's entry is in a closed group here
    const int32_t gslot = __shfl_sync(kFull, slot, myf < 0 ? 0 : myf);
    const bool mybad = gslot < 0 || static_cast<int64_t>(gslot) >= a.S;

    // the stream's rows and the chunk's token rows and snapshot rows (element pointers)
    GradT* const grad_s = static_cast<GradT*>(a.grad) + static_cast<int64_t>(cl) * a.S * hd;
    BankT* const bank_s = static_cast<BankT*>(a.bank) + static_cast<int64_t>(cl) * a.S * hd;
    const BankT* const snap_c = static_cast<const BankT*>(a.snap) + static_cast<int64_t>(cl) * nk * hd;
    const float* const dva_chunk = a.dva + c * a.C * static_cast<int64_t>(hd);
    uint32_t bad = 0;
    float dk = 0.f, gs = 0.f;   // this lane's entry: its <dva, snap> and <gdw, snap> sums over the slices
    if (cend >= f0) {
        for (int sl = 0; sl < a.nsl; ++sl) {
            const int col = sl * 128 + lane * 4;
            const bool on = col < hd;
            const int ccol = on ? col : 0;   // a lane past the row copies nothing (zero fill) from column 0
            // position k's rows go to ring slot (k - f0) % kPaRing: its token row, and for a group's
            // FIRST the group's grad and snapshot rows; one commit group per position
            auto issue = [&](int k) {
                if (k <= cend) {   // warp-uniform
                    const int ks = (k - f0) & (kPaRing - 1);
                    const int tk = __shfl_sync(kFull, t, k);
                    const int32_t sk = __shfl_sync(kFull, slot, k);
                    if ((okmask >> k) & 1u)
                        cp4z(reinterpret_cast<float*>(&ring.dva[ks][lane]), dva_chunk + tk * hd + ccol, on);
                    if (((fmask >> k) & 1u) && sk >= 0 && static_cast<int64_t>(sk) < a.S) {
                        const int g = ord0 + __popc(fmask & ((1u << k) - 1u));
                        cp4z(&ring.grad[ks][lane][0], grad_s + static_cast<int64_t>(sk) * hd + ccol, on);
                        cp4z(&ring.snap[ks][lane][0], snap_c + static_cast<int64_t>(g) * hd + ccol, on);
                    }
                }
                cp_commit();
            };
#pragma unroll 1
            for (int k = f0; k < f0 + kPaRing - 1; ++k) issue(k);
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, cg[4] = {0.f, 0.f, 0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
            int64_t crow = 0;
            bool cbad = true;
            float gfirst = 0.f;   // a FIRST lane: its group's <gdw, snap> over this slice
            // positions in aligned blocks of 8: the block's dot partials are reduced across the lanes
            // together (transposed), position k's sum landing in lane k
#pragma unroll 1
            for (int blk = f0 >> 3; blk <= (cend >> 3); ++blk) {
                float dp[8], gp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    dp[i] = 0.f;
                    gp[i] = 0.f;
                    const int k = blk * 8 + i;
                    if (k < f0 || k > cend) continue;   // warp-uniform
                    issue(k + kPaRing - 1);
                    cp_wait<kPaRing - 1>();   // position k's copies have landed (zeros past the row)
                    const int ks = (k - f0) & (kPaRing - 1);
                    if ((fmask >> k) & 1u) {    // a group starts: its rows become current
                        const int32_t sk = __shfl_sync(kFull, slot, k);
                        cbad = sk < 0 || static_cast<int64_t>(sk) >= a.S;
                        crow = static_cast<int64_t>(cbad ? 0 : sk) * hd + ccol;
#pragma unroll
                        for (int x = 0; x < 4; ++x) acc[x] = 0.f;
                        if (!cbad) {
                            get4(&ring.grad[ks][lane][0], cg);
                            get4(&ring.snap[ks][lane][0], cs);
                            if (on) copy_raw4(bank_s + crow, &ring.snap[ks][lane][0]);
                            gp[i] = dot4(cg, cs);
                        } else {
                            bad = 1u;
                        }
                    }
                    const float skk = __shfl_sync(kFull, sc, k);
                    if (!cbad && ((okmask >> k) & 1u)) {
                        float d[4];
                        get4(reinterpret_cast<const float*>(&ring.dva[ks][lane]), d);
#pragma unroll
                        for (int x = 0; x < 4; ++x) acc[x] = fmaf(skk, d[x], acc[x]);
                        dp[i] = dot4(d, cs);
                    }
                    if ((lmask >> k) & 1u) {    // the group ends: its grad row
                        const float cpl = __shfl_sync(kFull, cp, k);
                        if (!cbad && on) {
                            float ov[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) ov[x] = fmaf(cg[x], cpl, acc[x]);
                            st4(grad_s + crow, ov);
                        }
                    }
                }
                // index (lane & 15) of the 16 values ends in lane `lane`: the block's entry dots sit at
                // i + 8 * (blk & 1) so that position 8 * blk + i is lane-aligned, the group dots at the other half
                const bool odd = (blk & 1) != 0;
                float vals[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    vals[i] = odd ? gp[i] : dp[i];
                    vals[i + 8] = odd ? dp[i] : gp[i];
                }
                const float red = tsum16(vals, lane);
                const float gred = __shfl_xor_sync(kFull, red, 8);
                const bool inblk = (lane >> 3) == blk && lane >= f0 && lane <= cend;
                if (inblk) {
                    dk += red;
                    if ((fmask >> lane) & 1u) gfirst = gred;
                }
            }
            // every member adds its group's <gdw, snap> (from the group's FIRST lane)
            const float g_of_mine = __shfl_sync(kFull, gfirst, myf < 0 ? 0 : myf);
            if (myf >= 0) gs += g_of_mine;
            cp_wait<0>();
        }
        if (mine) {
            a.d_k_eff[o] = mybad ? 0.f : -be * dk;
            a.grad_g[o] = mybad ? 0.f : cp * gs;
        }
    }
    // the walk reuses the warp's ring (idle by now: every copy has landed) as kWalkRows token-row slots
    if (open)
        open_group<GradT, BankT, ValT>(a, srow, c, cl, q0 + flast, ord0 + __popc(fmask) - 1, lane, &bad, &wsm.walk[0][0]);
    if (bad && lane == 0 && a.status != nullptr) atomicOr(a.status, kDevBadSlot);
}

template <typename GradT, typename BankT, typename ValT>
cudaError_t launch_t(const PAArgs& a, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>(a.P) * static_cast<unsigned>(a.tiles);
    constexpr size_t smem = pa_smem_bytes<GradT, BankT>();
    cudaError_t e = cudaFuncSetAttribute(pa_kernel<GradT, BankT, ValT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_dependent(pa_kernel<GradT, BankT, ValT>, dim3(blocks), dim3(kPaThreads), smem, stream, a);
}

template <typename GradT, typename BankT>
cudaError_t launch_v(const PAArgs& a, int val_bf16, cudaStream_t stream) {
    return val_bf16 ? launch_t<GradT, BankT, __nv_bfloat16>(a, stream) : launch_t<GradT, BankT, float>(a, stream);
}

cudaError_t launch_pa(const PAArgs& a, int grad_bf16, int bank_bf16, int val_bf16, cudaStream_t stream) {
    if (grad_bf16)
        return bank_bf16 ? launch_v<__nv_bfloat16, __nv_bfloat16>(a, val_bf16, stream)
                         : launch_v<__nv_bfloat16, float>(a, val_bf16, stream);
    return bank_bf16 ? launch_v<float, __nv_bfloat16>(a, val_bf16, stream) : launch_v<float, float>(a, val_bf16, stream);
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" sdm_status sdm_pa(const sdm_shape* shape, int32_t grad_dtype, const int32_t* sorted_k, const int32_t* k_idx,
                             const void* k_val, const float* log_k, const void* cpe, const float* beta,
                             const float* dva, void* grad, void* bank, const void* snap, float* d_k_eff,
                             float* grad_g, int64_t step_begin, int64_t step_end, uint32_t* status,
                             sdm_stream_t stream) {
    const void* const ptrs[] = {sorted_k, k_idx, k_val, log_k, cpe, beta, dva, grad, bank, snap, d_k_eff, grad_g};
    const sdm_status st = checks::check_backward(shape, grad_dtype, step_begin, step_end, ptrs);
    if (st != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    PAArgs a;
    memset(&a, 0, sizeof(a));
    a.sorted_k = sorted_k;
    a.k_idx = k_idx;
    a.k_val = k_val;
    a.log_k = log_k;
    a.cpe = cpe;
    a.beta = beta;
    a.dva = dva;
    a.grad = grad;
    a.bank = bank;
    a.d_k_eff = d_k_eff;
    a.grad_g = grad_g;
    a.status = status;
    a.P = shape->P;
    a.C = shape->C;
    a.W = shape->W;
    a.nk = shape->C * shape->W;
    a.hd = shape->hd;
    a.nsl = (shape->hd + 127) / 128;
    a.tiles = (a.nk + kPaTile - 1) / kPaTile;
    a.S = shape->S;
    const size_t bank_elem = shape->bank_dtype == SDM_BF16 ? 2 : 4;
    const int64_t step_rows = static_cast<int64_t>(a.P) * a.nk;   // snapshot rows of one step
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // the backward runs the steps last to first: step ti reads the grad rows step ti + 1 wrote
    for (int64_t ti = step_end - 1; ti >= step_begin; --ti) {
        a.c0 = ti * a.P;
        a.snap = static_cast<const unsigned char*>(snap) + (ti - step_begin) * step_rows * a.hd * bank_elem;
        if (launch_pa(a, grad_dtype == SDM_BF16, shape->bank_dtype == SDM_BF16, shape->val_dtype == SDM_BF16, cs) !=
            cudaSuccess)
            return SDM_ERR_CUDA;
    }
    return SDM_OK;
}
