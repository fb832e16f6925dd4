// sdm_phase1.cu -- Phase 1 of the chunked sparse-delta-memory forward, one CTA per chunk, on chip.
//
// What it computes (sparse-delta-memory 2.0.0, phase1_cuda.py: module docstring,
// p1_keys_zw_kernel, p1_scan_kernel, p1_pairs_kernel comment): the chunk's write (K) and read (Q)
// entries are sorted stably by slot; per slot group, the log-cumsum of the gates (a write entry's
// gate counts once per token: a token's repeated write entry adds 0), rex = gates after the
// entry, cpe = exp(group total) in the value type, the flags, the packed positions and the sorted
// rows; then the pair triangles A (write x earlier write of another token) and QK (read x
// earlier write, own token included). It also writes the DW records of the chunk's sorted write
// row, partitioned into hashed slot buckets (the DW kernel's work split), with each bucket's start.
//
// GB300 design (not the pages' kernels): the whole chunk (up to 8192 entries) stays in shared
// memory from load to the last output byte:
//   0. load ids, values and gates (coalesced, all of a thread's loads in flight together) into
//      entry-indexed arrays;
//   1. stable sort of entry indices by slot: a counting sort by the key's top bits (shared-memory
//      bucket counts, one block scan, an atomic scatter, then each entry ranks itself inside its
//      bucket by (key, entry)), or, when a bucket is crowded (skewed slots), an LSD radix sort in
//      4-bit digits with per-thread digit counters;
//   2. a forward and a reverse segmented block scan with TwoSum-compensated f32 sums (fixed
//      tree: bitwise reproducible), emitting the per-entry results into entry-indexed arrays and a
//      word per write-row position; one pass over the write row then writes the sorted write row
//      and the DW records, partitioned into hashed slot buckets;
//   3. every entry-order output written from shared memory by consecutive threads (4 entries per
//      thread, vector loads and stores, when W and R are multiples of 4);
//   4. pair triangles: A and QK are zero-filled by 16-byte L1-bypassing stores of every thread, paced
//      by the SM clock over phases 0-3 (a steady stream under the compute); then one warp per
//      (row, triangle) walks: 32 earlier positions per step, lanes of one cell summed by a fixed
//      shuffle tree, one lane adds the cell's partial to the warp's row buffer; only rows with
//      terms are rewritten.
#include <cuda_bf16.h>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ uint32_t lanemask_le() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_le;" : "=r"(m));
    return m;
}

// ---- compensated segmented-scan elements ------------------------------------------------------
// Forward element: the sum (s + c) and the valid K / Q counts of the LAST segment of the range
// (cnt: K in bits 0..15, Q in bits 16..30), the unsegmented K / Q entry counts (allh: K in
// 0..15, Q in 16..30) and, in allh bit 31, whether a segment (group) starts inside the range.
struct Fwd {
    float s, c;
    uint32_t cnt, allh;
};
// Reverse element (the reversed sequence): the same sum and counts of the range's last segment
// in reversed order, cnt bit 31 = a group's last entry lies inside the range, and tot = the
// log-cumsum at that last entry (the group total).
struct Bwd {
    float s, c;
    uint32_t cnt;
    float tot;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// a precedes b
__device__ __forceinline__ Fwd fcomb(const Fwd& a, const Fwd& b) {
    const uint32_t all = (a.allh & 0x7FFFFFFFu) + (b.allh & 0x7FFFFFFFu);
    Fwd r;
    if (b.allh >> 31) {
        r.s = b.s;
        r.c = b.c;
        r.cnt = b.cnt;
        r.allh = all | 0x80000000u;
    } else {
        float err;
        two_sum(a.s, b.s, r.s, err);
        r.c = __fadd_rn(__fadd_rn(a.c, b.c), err);
        r.cnt = a.cnt + b.cnt;
        r.allh = all | (a.allh & 0x80000000u);
    }
    return r;
}

// A precedes B in the reversed order (A holds later positions)
__device__ __forceinline__ Bwd bcomb(const Bwd& A, const Bwd& B) {
    if (B.cnt >> 31) return B;
    Bwd r;
    float err;
    two_sum(A.s, B.s, r.s, err);
    r.c = __fadd_rn(__fadd_rn(A.c, B.c), err);
    r.cnt = ((A.cnt & 0x7FFFFFFFu) + B.cnt) | (A.cnt & 0x80000000u);
    r.tot = A.tot;
    return r;
}

__device__ __forceinline__ Fwd shfl_up_f(const Fwd& v, int d) {
    return {__shfl_up_sync(kFull, v.s, d), __shfl_up_sync(kFull, v.c, d), __shfl_up_sync(kFull, v.cnt, d),
            __shfl_up_sync(kFull, v.allh, d)};
}
__device__ __forceinline__ Bwd shfl_down_b(const Bwd& v, int d) {
    return {__shfl_down_sync(kFull, v.s, d), __shfl_down_sync(kFull, v.c, d), __shfl_down_sync(kFull, v.cnt, d),
            __shfl_down_sync(kFull, v.tot, d)};
}

// Exclusive prefix (aggregate of every earlier thread) of the threads' aggregates, forward.
// scr: 64 elements of scratch. Contains two block barriers.
__device__ __noinline__ Fwd fwd_block_prefix(Fwd x, Fwd* scr, int lane, int warp, int nw) {
    const Fwd zero = {0.f, 0.f, 0u, 0u};
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Fwd y = shfl_up_f(x, d);
        if (lane >= d) x = fcomb(y, x);
    }
    if (lane == 31) scr[warp] = x;
    __syncthreads();
    if (warp == 0) {
        Fwd w = lane < nw ? scr[lane] : zero;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const Fwd y = shfl_up_f(w, d);
            if (lane >= d) w = fcomb(y, w);
        }
        Fwd ex = shfl_up_f(w, 1);
        if (lane == 0) ex = zero;
        if (lane < nw) scr[32 + lane] = ex;
    }
    __syncthreads();
    Fwd lx = shfl_up_f(x, 1);
    if (lane == 0) lx = zero;
    return fcomb(scr[32 + warp], lx);
}

// Exclusive prefix in the reversed order (aggregate of every later thread).
__device__ __noinline__ Bwd bwd_block_prefix(Bwd x, Bwd* scr, int lane, int warp, int nw) {
    const Bwd zero = {0.f, 0.f, 0u, 0.f};
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const Bwd y = shfl_down_b(x, d);
        if (lane + d < 32) x = bcomb(y, x);
    }
    if (lane == 0) scr[warp] = x;
    __syncthreads();
    if (warp == 0) {
        Bwd w = lane < nw ? scr[lane] : zero;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const Bwd y = shfl_down_b(w, d);
            if (lane + d < nw) w = bcomb(y, w);
        }
        Bwd ex = shfl_down_b(w, 1);
        if (lane == nw - 1) ex = zero;
        if (lane < nw) scr[32 + lane] = ex;
    }
    __syncthreads();
    Bwd lx = shfl_down_b(x, 1);
    if (lane == 31) lx = zero;
    return bcomb(scr[32 + warp], lx);
}

// In-place exclusive scan (block-wide) of cnt counters stored with one padding word after every
// `group` of them: logical index i lives at a[i + i / group].
// In-place exclusive scan (block-wide) of cnt counters stored with one padding slot after every
// `group` of them: logical index i lives at a[i + i / group]. Each thread takes a contiguous run of
// logical indices and walks the padded addresses incrementally (one division per thread).
template <typename T>
__device__ __noinline__ void block_exscan_padded(T* a, int cnt, int group, uint32_t* scr, int lane, int warp, int nw) {
    const int per = (cnt + blockDim.x - 1) / blockDim.x;
    const int i0 = threadIdx.x * per;
    const int n_mine = max(0, min(per, cnt - i0));
    const int r0 = i0 / group;
    const int start = i0 + r0;               // padded address of i0
    const int left0 = group - (i0 - r0 * group);   // entries left in the first row
    uint32_t s = 0;
    {
        int addr = start, left = left0;
        for (int j = 0; j < n_mine; ++j) {
            s += a[addr];
            ++addr;
            if (--left == 0) {
                ++addr;   // skip the padding slot
                left = group;
            }
        }
    }
    uint32_t x = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) scr[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < nw ? scr[lane] : 0u;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, w, d);
            if (lane >= d) w += y;
        }
        if (lane < nw) scr[32 + lane] = w - (lane < nw ? scr[lane] : 0u);
    }
    __syncthreads();
    uint32_t acc = scr[32 + warp] + x - s;
    {
        int addr = start, left = left0;
        for (int j = 0; j < n_mine; ++j) {
            const uint32_t v = a[addr];
            a[addr] = static_cast<T>(acc);
            acc += v;
            ++addr;
            if (--left == 0) {
                ++addr;
                left = group;
            }
        }
    }
}

// A / QK of chunk c set to zero by the block with plain stores (the triangles are not a whole
// number of 16-byte units, so the TMA bulk fill does not apply). Out of line: rarely used.
__device__ __noinline__ void zero_triangles(float* A, float* QK, int64_t c, int64_t cells) {
    for (int m = 0; m < 2; ++m) {
        float* const base = m == 0 ? A : QK;
        if (base == nullptr) continue;
        float* const chunk = base + c * cells;
        for (int64_t i = threadIdx.x; i < cells; i += blockDim.x) __stcs(chunk + i, 0.f);
    }
}

// Global stores of Phase 1 bypass L1 (L1::no_allocate): the stores of a chunk (its outputs, 512 KB of
// zeros, its DW records) would otherwise evict the lines its spills and loads use. Measured on the
// large workload: with the streaming hint instead 2 us slower per Phase 1; plain write-back stores of
// the zeros 70 us slower.
__device__ __forceinline__ void st_na(float* p, float v) { asm volatile("st.global.L1::no_allocate.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory"); }
__device__ __forceinline__ void st_na(int32_t* p, int32_t v) { asm volatile("st.global.L1::no_allocate.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory"); }
__device__ __forceinline__ void st_na(int8_t* p, int8_t v) { asm volatile("st.global.L1::no_allocate.s8 [%0], %1;" ::"l"(p), "r"(static_cast<int>(v)) : "memory"); }
__device__ __forceinline__ void st_na(__nv_bfloat16* p, __nv_bfloat16 v) {
    asm volatile("st.global.L1::no_allocate.b16 [%0], %1;" ::"l"(p), "h"(__bfloat16_as_ushort(v)) : "memory");
}
__device__ __forceinline__ void st_na(int4* p, int4 v) {
    asm volatile("st.global.L1::no_allocate.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_na(float4* p, float4 v) {
    asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ void st_na(uint4* p, uint4 v) {
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_na(uint2* p, uint2 v) {
    asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_na(uint32_t* p, uint32_t v) {
    asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
template <typename T>
__device__ __forceinline__ void st_stream(T* p, T v) {
    st_na(p, v);
}

// Four consecutive values of the value type: loaded from shared memory as one vector (8 bytes for
// bfloat16, 16 for float32), stored to global memory as one vector store (L1 bypassed).
__device__ __forceinline__ void ld4(const float* p, float (&v)[4]) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(x.x << 16); v[1] = __uint_as_float(x.x & 0xFFFF0000u);
    v[2] = __uint_as_float(x.y << 16); v[3] = __uint_as_float(x.y & 0xFFFF0000u);
}
__device__ __forceinline__ void st4(float* p, const float (&v)[4]) {
    st_na(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float (&v)[4]) {
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[0]))) |
                        static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[1]))) << 16;
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2]))) |
                        static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[3]))) << 16;
    st_na(reinterpret_cast<uint2*>(p), make_uint2(lo, hi));
}
// Four int8 flags packed into one 4-byte store.
__device__ __forceinline__ void st4_flags(int8_t* p, uint32_t f0, uint32_t f1, uint32_t f2, uint32_t f3) {
    st_na(reinterpret_cast<uint32_t*>(p), f0 | f1 << 8 | f2 << 16 | f3 << 24);
}

// ORD: the saving forward's Phase 1 -- each group's FIRST record also carries its dense ordinal
// and out.ngroups is written (a separate instantiation: the plain forward's kernel is unchanged)
template <typename ValT, bool ORD>
__global__ void __launch_bounds__(kMaxThreads, 1) p1_kernel(const P1Args a) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* const keys = reinterpret_cast<uint32_t*>(smem + a.sm_keys);   // entry -> key word
    ValT* const vals = reinterpret_cast<ValT*>(smem + a.sm_vals);          // entry -> value
    uint16_t* const sidx = reinterpret_cast<uint16_t*>(smem + a.sm_sidx);  // sorted position -> entry
    float* const lv = reinterpret_cast<float*>(smem + a.sm_lv);            // entry -> log-cumsum
    uint32_t* const posv = reinterpret_cast<uint32_t*>(smem + a.sm_pos);   // entry -> position pack
    uint16_t* const kbv = reinterpret_cast<uint16_t*>(smem + a.sm_kb);     // entry -> K entries before
    float* const rexv = reinterpret_cast<float*>(smem + a.sm_rex);         // write entry o -> rex
    float* const cpev = reinterpret_cast<float*>(smem + a.sm_tot);         // write entry o -> cpe (value type)
    // write-row index -> entry | (FIRST: group size, then the group's record base) << 16
    uint32_t* const krpos = reinterpret_cast<uint32_t*>(smem + a.sm_kslot);
    uint32_t* const bcnt = reinterpret_cast<uint32_t*>(smem + a.sm_bcnt);  // [B + 1] sizes / offsets | [B] fill
    Fwd* const fscr = reinterpret_cast<Fwd*>(smem + a.sm_scr);
    Bwd* const bscr = reinterpret_cast<Bwd*>(smem + a.sm_scr);
    uint32_t* const uscr = reinterpret_cast<uint32_t*>(smem + a.sm_scr + 64 * sizeof(Fwd));

    // rows (token) of A (0) / QK (1) with at least one entry that has an earlier write entry in
    // its group: only these rows have terms
    __shared__ uint32_t rowmask[2][kMaxC / 32];
    // sorted positions of the first write entry of each slot group with >= kHotMin write entries:
    // the candidates for the dense pair path
    __shared__ uint32_t hotmask[kMaxRow / 32];
    __shared__ int hot_n;
    __shared__ uint32_t row_claim;   // the next flagged (triangle, row) pair to take (phase 4)
    // per (triangle, token): the dense groups with a term in the token's A (0) / QK (1) row
    __shared__ uint32_t hotrow[2][kMaxC];
    // write-row positions of the valid write groups' first entries, a bit per position: the dense
    // ordinal of a group = the heads before it
    __shared__ uint32_t khead[kMaxRow / 32];
    // long groups: count and tail fill
    __shared__ uint32_t lcnt_s, ltail_s;
    __shared__ uint32_t ngroups_s;   // valid write groups (out.stats)
    // the long-group kernel that follows may be scheduled once every CTA of this grid runs (it waits
    // for this grid's completion before it reads anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        lcnt_s = 0u;
        ngroups_s = 0u;
        ltail_s = 0u;
        row_claim = 0u;
    }
    const int nw = a.nwarps, nthr = blockDim.x;
    if (tid < 2 * (kMaxC / 32)) rowmask[tid / (kMaxC / 32)][tid % (kMaxC / 32)] = 0u;
    for (int i = tid; i < kMaxRow / 32; i += blockDim.x) hotmask[i] = 0u;
    if constexpr (ORD)
        for (int i = tid; i < kMaxRow / 32; i += blockDim.x) khead[i] = 0u;
    for (int i = tid; i < 2 * kMaxC; i += blockDim.x) hotrow[i / kMaxC][i % kMaxC] = 0u;
    const int nbk = 1 << a.logB;   // DW buckets per stream (their counters are zeroed after the sort)
    // A and QK start as zeros (16-byte stores spread over the phases when the chunk's triangles are
    // a whole number of 16-byte units, else plain stores at the start); rows with terms are
    // rewritten at the end.
    const int64_t cells = static_cast<int64_t>(a.C) * a.C;
    const bool bulk_zero = (cells & 3) == 0 && (a.out.A != nullptr || a.out.QK != nullptr);
    auto bucket_of = [&](uint32_t key) -> uint32_t {
        return a.logB == 0 ? 0u : (key * 0x9E3779B1u) >> (32 - a.logB);
    };
    const int64_t c = a.c0 + blockIdx.x;
    const int C = a.C, W = a.W, R = a.R, wr = a.wr, n = a.n, nk = a.nk, nq = a.nq, npad = a.npad;
    const int V = c >= a.first_partial ? a.valid_last : C;
    const uint32_t kmax = (a.key_bits >= 31) ? 0x7FFFFFFFu : ((1u << a.key_bits) - 1u);
    const ValT* kv = static_cast<const ValT*>(a.k_val) + c * nk;
    const ValT* qv = static_cast<const ValT*>(a.q_val) + c * nq;
    const int32_t* kid = a.k_idx + c * nk;
    const int32_t* qid = a.q_idx + c * nq;
    const float* gch = a.g + c * C * a.g_width;

    // ---- 0. load: every id and value of the chunk, all loads of a thread in flight together; the
    // chunk's gates go to the rex region (idle until the reverse scan; the LSD sort's counters, where
    // they lie over it, bring them back after the sort)
    float* const gs = rexv;
    const int ngate = C * a.g_width;
    auto load_gates = [&]() {
        for (int i = tid; i < ngate; i += nthr) gs[i] = __ldg(gch + i);
    };
    load_gates();
    {
        bool bad = false;
        const int total = nk + nq;
        for (int i0 = tid; i0 < total; i0 += kItems * nthr) {
            int32_t id[kItems];
            ValT vv[kItems];
#pragma unroll
            for (int u = 0; u < kItems; ++u) {
                const int i = i0 + u * nthr;
                if (i < nk) {
                    id[u] = __ldg(kid + i);
                    vv[u] = kv[i];
                } else if (i < total) {
                    id[u] = __ldg(qid + (i - nk));
                    vv[u] = qv[i - nk];
                }
            }
#pragma unroll
            for (int u = 0; u < kItems; ++u) {
                const int i = i0 + u * nthr;
                if (i < total) {
                    const bool isq = i >= nk;
                    const int o = isq ? i - nk : i;
                    const int lanes = isq ? R : W;
                    const int t = static_cast<int>(__umulhi(static_cast<uint32_t>(o), isq ? a.r_magic : a.w_magic));
                    const int ln = o - t * lanes;
                    const int e = t * wr + (isq ? W : 0) + ln;
                    uint32_t key = kmax | kKeyInvalid;
                    ValT v = from_f<ValT>(0.f);
                    if (t < V) {
                        if (id[u] >= 0 && static_cast<int64_t>(id[u]) < a.S) {
                            key = static_cast<uint32_t>(id[u]);
                            v = vv[u];
                        } else {
                            bad = true;
                        }
                    }
                    keys[e] = key;
                    vals[e] = v;
                }
            }
        }
        for (int e = n + tid; e < npad; e += nthr) {
            keys[e] = kmax | kKeyInvalid;
            vals[e] = from_f<ValT>(0.f);
        }
        if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, kDevBadSlot);
    }
    if (!bulk_zero && (a.out.A != nullptr || a.out.QK != nullptr)) zero_triangles(a.out.A, a.out.QK, c, cells);
    {   // the counting sort's bucket counts start at zero
        uint32_t* const bc = reinterpret_cast<uint32_t*>(smem + a.sm_pos);
        for (int b = tid; b < (1 << a.bucket_bits); b += nthr) bc[b] = 0u;
    }
    __syncthreads();
    // A and QK of the chunk start as zeros written by every thread with 16-byte stores (L1 bypassed),
    // paced by the SM clock: a warp stores one unit per thread each kZeroPeriod cycles (the warps
    // a 1/32 period apart), checked once per item in the per-item loops below. The stores so form
    // a steady stream under the block's compute; issued in bursts at the phase boundaries they
    // stalled the block (about 20 us more per Phase 1 on the large workload). Rows with terms are
    // written again in phase 4, after the flush of the units left and a block barrier. Thread
    // tid's units of a triangle are tid, tid + nthr, ... (A's, then QK's).
    const int zper_m = bulk_zero ? static_cast<int>(cells / 4) : 0;   // 16-byte units per triangle
    const int zka = a.out.A != nullptr && zper_m > tid ? (zper_m - tid + nthr - 1) / nthr : 0;
    const int zkq = a.out.QK != nullptr && zper_m > tid ? (zper_m - tid + nthr - 1) / nthr : 0;
    float* const za = a.out.A != nullptr ? a.out.A + c * cells + static_cast<int64_t>(tid) * 4 : nullptr;
    float* const zq = a.out.QK != nullptr ? a.out.QK + c * cells + static_cast<int64_t>(tid) * 4 : nullptr;
    const int zstride = nthr * 4;
    int zero_next = 0;   // this thread's next unit
    uint32_t zdl = static_cast<uint32_t>(clock()) + static_cast<uint32_t>(warp) * (kZeroPeriod / 32u);
    auto zero_store = [&]() {
        float* const p = zero_next < zka ? za + zero_next * zstride : zq + (zero_next - zka) * zstride;
        st_na(reinterpret_cast<float4*>(p), make_float4(0.f, 0.f, 0.f, 0.f));
        ++zero_next;
    };
    auto zpace = [&]() {   // one unit when this warp's next time has come
        if (zero_next < zka + zkq && static_cast<int32_t>(static_cast<uint32_t>(clock()) - zdl) >= 0) {
            zero_store();
            zdl += kZeroPeriod;
        }
    };
    zpace();

    // ---- 1. stable sort of the entries by key --------------------------------------------------
    // Fast path, a counting sort by the top bits of the key (the bucket): each valid entry counts
    // into its bucket with a shared atomic, one block scan turns the counts into bucket starts, each
    // entry takes a place in its bucket with a second atomic (in whatever order the atomics run),
    // and then every bucket's entries are ranked inside it by (key, entry), which is unique: the
    // result is the stable order whatever the atomics did. Invalid entries go after every valid one
    // in entry order. A chunk with a bucket of more than kBucketMax entries (skewed slots) takes the
    // LSD radix sort instead. The entries move as words: entry (13 bits) | the key's bits under
    // the bucket << 13.
    uint32_t* const bstart = reinterpret_cast<uint32_t*>(smem + a.sm_pos);   // [2^bbits] counts -> starts -> ends
    uint32_t* const bword = reinterpret_cast<uint32_t*>(smem + a.sm_pong);   // words by sorted position
    const int bbits = a.bucket_bits;   // <= key_bits, and 2^bbits <= npad: the counts fit their region
    const int bsh = a.key_bits - bbits;                                      // bucket = key >> bsh
    const int nbuck = 1 << bbits;
    bool fast;
    {
        const int p0 = tid * kItems;
        uint32_t kw[kItems];
        {
            const uint4 k0 = *reinterpret_cast<const uint4*>(keys + p0);
            const uint4 k1 = *reinterpret_cast<const uint4*>(keys + p0 + 4);
            kw[0] = k0.x; kw[1] = k0.y; kw[2] = k0.z; kw[3] = k0.w;
            kw[4] = k1.x; kw[5] = k1.y; kw[6] = k1.z; kw[7] = k1.w;
        }
        uint32_t ninv = 0;
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            if (kw[k] >> 31) ++ninv;
            else atomicAdd(&bstart[kw[k] >> bsh], 1u);
            zpace();
        }
        __syncthreads();
        // block scan of the counts: thread t owns buckets [bt0, bt1), a contiguous segment
        const int per = (nbuck + nthr - 1) / nthr;
        const int bt0 = min(nbuck, tid * per), bt1 = min(nbuck, bt0 + per);
        const bool vseg = per == 8 && bt1 - bt0 == 8;   // the usual case: two 16-byte loads
        uint32_t sv[8];
        uint32_t seg = 0;
        bool big = false;
        if (vseg) {
            const uint4 v0 = *reinterpret_cast<const uint4*>(bstart + bt0);
            const uint4 v1 = *reinterpret_cast<const uint4*>(bstart + bt0 + 4);
            sv[0] = v0.x; sv[1] = v0.y; sv[2] = v0.z; sv[3] = v0.w;
            sv[4] = v1.x; sv[5] = v1.y; sv[6] = v1.z; sv[7] = v1.w;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                seg += sv[q];
                big |= sv[q] > static_cast<uint32_t>(kBucketMax);
            }
        } else {
            for (int b = bt0; b < bt1; ++b) {
                const uint32_t v = bstart[b];
                seg += v;
                big |= v > static_cast<uint32_t>(kBucketMax);
            }
        }
        uint32_t xs = seg, xi = ninv;   // inclusive over the warp: bucket counts, invalid entries
#pragma unroll
        for (int dd = 1; dd < 32; dd <<= 1) {
            const uint32_t ys = __shfl_up_sync(kFull, xs, dd), yi = __shfl_up_sync(kFull, xi, dd);
            if (lane >= dd) {
                xs += ys;
                xi += yi;
            }
        }
        if (lane == 31) {
            uscr[warp] = xs;
            uscr[32 + warp] = xi;
        }
        fast = !__syncthreads_or(big);
        zpace();
        // every warp: the totals of the warps before it, and of all warps
        uint32_t ws = lane < nw ? uscr[lane] : 0u, wi = lane < nw ? uscr[32 + lane] : 0u;
        const uint32_t ws0 = ws, wi0 = wi;
#pragma unroll
        for (int dd = 1; dd < 32; dd <<= 1) {
            const uint32_t ys = __shfl_up_sync(kFull, ws, dd), yi = __shfl_up_sync(kFull, wi, dd);
            if (lane >= dd) {
                ws += ys;
                wi += yi;
            }
        }
        const uint32_t nvalid = __shfl_sync(kFull, ws, 31);
        const uint32_t s_before = __shfl_sync(kFull, ws - ws0, warp) + xs - seg;     // bucket entries before mine
        const uint32_t i_before = __shfl_sync(kFull, wi - wi0, warp) + xi - ninv;    // invalid entries before mine
        if (fast) {
            uint32_t run = s_before;
            if (vseg) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t v = sv[q];
                    sv[q] = run;
                    run += v;
                }
                *reinterpret_cast<uint4*>(bstart + bt0) = make_uint4(sv[0], sv[1], sv[2], sv[3]);
                *reinterpret_cast<uint4*>(bstart + bt0 + 4) = make_uint4(sv[4], sv[5], sv[6], sv[7]);
            } else {
                for (int b = bt0; b < bt1; ++b) {
                    const uint32_t v = bstart[b];
                    bstart[b] = run;
                    run += v;
                }
            }
        }
        __syncthreads();
        if (fast) {
            zpace();
            const uint32_t lowm = bsh > 0 ? (1u << bsh) - 1u : 0u;
            uint32_t ipos = nvalid + i_before;
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                zpace();
                const uint32_t e = static_cast<uint32_t>(p0 + k);
                if (kw[k] >> 31) {   // invalid: after every valid entry, in entry order (final)
                    if (ipos < static_cast<uint32_t>(npad)) sidx[ipos] = static_cast<uint16_t>(e);
                    ++ipos;
                } else {
                    const uint32_t pos = atomicAdd(&bstart[kw[k] >> bsh], 1u);   // bstart becomes the end
                    if (pos < static_cast<uint32_t>(npad)) bword[pos] = e | (kw[k] & lowm) << kSortWordEntryBits;
                }
            }
            __syncthreads();
            zpace();
            // each valid entry's place: the start of its bucket (the previous bucket's end) plus the
            // number of the bucket's words below its own (key bits under the bucket, then entry)
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                zpace();
                if (kw[k] >> 31) continue;
                const uint32_t e = static_cast<uint32_t>(p0 + k);
                const uint32_t b = kw[k] >> bsh;
                const uint32_t en = bstart[b];
                const uint32_t st = b > 0 ? bstart[b - 1] : 0u;
                uint32_t r = st;
                if (en - st > 1u) {
                    const uint32_t w = e | (kw[k] & lowm) << kSortWordEntryBits;
                    for (uint32_t j = st; j < en; ++j) r += bword[j] < w ? 1u : 0u;
                }
                if (r < static_cast<uint32_t>(npad)) sidx[r] = static_cast<uint16_t>(e);
            }
            __syncthreads();
        }
    }
    // Fallback: a stable LSD radix sort of entry indices by key (low key_bits bits), 4-bit digits.
    // Every thread ranks its kItems consecutive positions (p0 = tid * kItems ...) with its own digit
    // counters in shared memory, cnt[digit][thread] (uint16); one block scan of the counters in
    // (digit, thread) order -- each thread a segment of 16 consecutive counters -- turns them into
    // first positions; one scatter. Positions follow (digit, thread, item) order, which within a
    // digit is the position order: the sort is stable. The counters alternate between two arrays
    // so that the next pass's are cleared while this pass uses its own. Between passes a position
    // holds a word: the entry (13 bits) and, once they fit in the other 19, the key bits still to
    // sort, so later passes read their digits with the word instead of gathering the entry's key.
    if (!fast) {
        uint32_t* const wa = reinterpret_cast<uint32_t*>(smem + a.sm_pong);     // words after even passes
        uint32_t* const wb = reinterpret_cast<uint32_t*>(smem + a.sm_pos);      // words after odd passes
        uint16_t* const cnt0 = reinterpret_cast<uint16_t*>(smem + a.sm_hist);   // [digit][thread], twice
        uint32_t* const wtot = uscr;                                            // per-warp totals
        const int p0 = tid * kItems;
        const int ncnt = kSortDigits * nthr;
        {   // this thread's scan segment of the first pass's counters starts at zero
            uint4* const seg = reinterpret_cast<uint4*>(cnt0) + 2 * tid;
            seg[0] = make_uint4(0u, 0u, 0u, 0u);
            seg[1] = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncthreads();
#pragma unroll 1
        for (int pass = 0; pass < a.passes; ++pass) {
            const int sh = pass * kSortDigitBits;
            const int left = a.key_bits - sh - kSortDigitBits;   // key bits still to sort after this pass
            const uint32_t dmask = (1u << min(kSortDigitBits, a.key_bits - sh)) - 1u;
            const bool last = pass == a.passes - 1;              // the last pass writes sidx
            const bool src_packed = a.key_bits - sh <= kSortWordKeyBits;
            const bool dst_packed = left <= kSortWordKeyBits;
            const uint32_t rmask = left > 0 ? (1u << left) - 1u : 0u;
            const uint32_t* const src = (pass & 1) ? wa : wb;
            uint32_t* const dst = (pass & 1) ? wb : wa;
            uint16_t* const cnt = cnt0 + (pass & 1) * ncnt;        // this pass's counters (zero)
            uint16_t* const nxt = cnt0 + ((pass + 1) & 1) * ncnt;  // the next pass's
            zpace();
            uint32_t kr[kItems];   // the entries' key bits sh and up
            uint32_t wv[kItems];   // the words this thread's positions move
            if (pass == 0) {
                const uint4 k0 = *reinterpret_cast<const uint4*>(keys + p0);
                const uint4 k1 = *reinterpret_cast<const uint4*>(keys + p0 + 4);
                kr[0] = k0.x; kr[1] = k0.y; kr[2] = k0.z; kr[3] = k0.w;
                kr[4] = k1.x; kr[5] = k1.y; kr[6] = k1.z; kr[7] = k1.w;
#pragma unroll
                for (int k = 0; k < kItems; ++k) wv[k] = static_cast<uint32_t>(p0 + k);
            } else {
                const uint4 v0 = *reinterpret_cast<const uint4*>(src + p0);
                const uint4 v1 = *reinterpret_cast<const uint4*>(src + p0 + 4);
                wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
                wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
#pragma unroll
                for (int k = 0; k < kItems; ++k) {
                    kr[k] = src_packed ? wv[k] >> kSortWordEntryBits : keys[wv[k] & kSortWordEntryMask] >> sh;
                    wv[k] &= kSortWordEntryMask;
                }
            }
            // rank among this thread's earlier items of the same digit: its counter, then + 1
            uint32_t dn = 0u, rn = 0u;   // per item a nibble: digit, rank
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const uint32_t d = kr[k] & dmask;
                uint16_t* const cp = cnt + d * nthr + tid;
                const uint32_t r = *cp;
                *cp = static_cast<uint16_t>(r + 1u);
                dn |= d << (4 * k);
                rn |= r << (4 * k);
                // the word this position moves: the entry and, packed, the key bits after this digit
                if (!last && dst_packed) wv[k] |= ((kr[k] >> kSortDigitBits) & rmask) << kSortWordEntryBits;
            }
            {   // clear this thread's segment of the next pass's counters (their last reader was the
                // previous pass's scatter, before its closing barrier)
                uint4* const seg = reinterpret_cast<uint4*>(nxt + kSortDigits * tid);
                seg[0] = make_uint4(0u, 0u, 0u, 0u);
                seg[1] = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
            zpace();
            // block scan of the counters in (digit, thread) order: this thread's segment holds the
            // counters [16 tid, 16 tid + 16), two per word
            uint4* const seg = reinterpret_cast<uint4*>(cnt + kSortDigits * tid);
            uint32_t sw[8];
            {
                const uint4 s0 = seg[0], s1 = seg[1];
                sw[0] = s0.x; sw[1] = s0.y; sw[2] = s0.z; sw[3] = s0.w;
                sw[4] = s1.x; sw[5] = s1.y; sw[6] = s1.z; sw[7] = s1.w;
            }
            uint32_t run = 0;   // exclusive prefixes within the segment (sums < 2^16: no carries)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t lo = sw[j] & 0xFFFFu, hi = sw[j] >> 16;
                sw[j] = run | (run + lo) << 16;
                run += lo + hi;
            }
            uint32_t x = run;
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, x, dd);
                if (lane >= dd) x += y;
            }
            if (lane == 31) wtot[warp] = x;
            __syncthreads();
            {   // every warp: the totals of the warps before it
                const uint32_t t = lane < nw ? wtot[lane] : 0u;
                uint32_t y = t;
#pragma unroll
                for (int dd = 1; dd < 32; dd <<= 1) {
                    const uint32_t z = __shfl_up_sync(kFull, y, dd);
                    if (lane >= dd) y += z;
                }
                const uint32_t off = __shfl_sync(kFull, y - t, warp) + x - run;   // before this segment
                const uint32_t o2 = off | off << 16;
                seg[0] = make_uint4(sw[0] + o2, sw[1] + o2, sw[2] + o2, sw[3] + o2);
                seg[1] = make_uint4(sw[4] + o2, sw[5] + o2, sw[6] + o2, sw[7] + o2);
            }
            __syncthreads();
            zpace();
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const uint32_t d = (dn >> (4 * k)) & 15u;
                const uint32_t pos = static_cast<uint32_t>(cnt[d * nthr + tid]) + ((rn >> (4 * k)) & 15u);
                if (pos < static_cast<uint32_t>(npad)) {
                    if (last)
                        sidx[pos] = static_cast<uint16_t>(wv[k]);
                    else
                        dst[pos] = wv[k];
                }
            }
            __syncthreads();
        }
        load_gates();   // the counters may have covered them
        __syncthreads();
    }
    // the DW bucket counters lay under the sort's digit counters: zeroed now, ordered before their
    // first use (the reverse scan) by the forward scan's barriers
    for (int b = tid; b < 2 * nbk + 1; b += nthr) bcnt[b] = 0u;

    // ---- 2. segmented scans over the sorted row -------------------------------------------------
    const int r0 = tid * kItems;
    uint32_t ke[kItems];   // entry at each of this thread's sorted positions (one 16-byte load)
    {
        const uint4 v = *reinterpret_cast<const uint4*>(sidx + r0);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < kItems; ++k) ke[k] = (w4[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
    }
    auto tok_of = [&](uint32_t e) { return __umulhi(e, a.wr_magic); };
    auto is_q_of = [&](uint32_t e) { return static_cast<int>(e - tok_of(e) * wr) >= W; };
    // head / tail bits, gates (a token's repeated write entry of a group adds 0)
    uint32_t headm = 0, tailm = 0, validm = 0, qm = 0, padm = 0;
    float x[kItems];
    uint32_t repc = 0;
    {
        uint32_t pk = kKeyInvalid, pe = 0;
        if (r0 > 0) {
            pe = sidx[r0 - 1];
            pk = keys[pe];
        }
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            zpace();
            const uint32_t e = ke[k], key = keys[e];
            const bool inv = key >> 31, pinv = pk >> 31;
            const bool head = (r0 + k == 0) || inv || pinv || (key != pk);
            headm |= (head ? 1u : 0u) << k;
            if (k > 0) tailm |= (head ? 1u : 0u) << (k - 1);
            const uint32_t t = tok_of(e);
            const int j = static_cast<int>(e - t * wr);
            const bool isq = j >= W;
            validm |= (inv ? 0u : 1u) << k;
            qm |= (isq ? 1u : 0u) << k;
            padm |= (e >= static_cast<uint32_t>(n) ? 1u : 0u) << k;
            const bool rep = !head && !isq && !is_q_of(pe) && tok_of(pe) == t;
            repc += rep ? 1u : 0u;
            x[k] = (!inv && !isq && !rep) ? gs[t * a.g_width + j * a.g_lane_stride] : 0.f;
            pk = key;
            pe = e;
        }
        // the last item ends its group when the next position starts one
        const uint32_t nkey = r0 + kItems < npad ? keys[sidx[r0 + kItems]] : kKeyInvalid;
        const bool tail = (pk >> 31) || (nkey >> 31) || (nkey != pk);
        tailm |= (tail ? 1u : 0u) << (kItems - 1);
    }
    // valid K / Q counts, and non-padding K / Q counts (kind-row indices)
    auto cnt_of = [&](int k) -> uint32_t {
        if (!((validm >> k) & 1u)) return 0u;
        return ((qm >> k) & 1u) ? (1u << 16) : 1u;
    };
    auto all_of = [&](int k) -> uint32_t {
        if ((padm >> k) & 1u) return 0u;
        return ((qm >> k) & 1u) ? (1u << 16) : 1u;
    };

    // forward: inclusive log-cumsum (lv, by entry); valid K entries before (kbv); own-kind peers
    // before and the index in the own kind's row, packed as before | index << 16 (both < 2^14), held
    // in posv until the reverse pass replaces it with the position pack
    {
        Fwd agg = {0.f, 0.f, 0u, 0u};
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            const Fwd it = {x[k], 0.f, cnt_of(k), all_of(k) | (((headm >> k) & 1u) << 31)};
            agg = k == 0 ? it : fcomb(agg, it);
        }
        Fwd run = fwd_block_prefix(agg, fscr, lane, warp, nw);
        zpace();
        // unrolled (measured 5 us faster per Phase 1 on the large workload than a rolled loop that
        // shifts the arrays; the reverse loop, four times larger, stays rolled)
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            zpace();
            const float xk = x[k];
            const uint32_t e = ke[k];
            const uint32_t ownc = cnt_of(k), owna = all_of(k);
            const Fwd it = {xk, 0.f, ownc, owna | (((headm >> k) & 1u) << 31)};
            run = fcomb(run, it);
            const float logv = __fadd_rn(run.s, run.c);
            const uint32_t b = run.cnt - ownc;   // valid K before | valid Q before << 16
            const uint32_t ex = (run.allh & 0x7FFFFFFFu) - owna;
            const bool isq = (qm >> k) & 1u;
            const uint32_t own_b = isq ? (b >> 16) : (b & 0xFFFFu);
            const uint32_t jxv = isq ? (ex >> 16) : (ex & 0xFFFFu);
            const bool valid = (validm >> k) & 1u;
            posv[e] = own_b | jxv << 16;
            lv[e] = valid ? logv : 0.f;
            const uint32_t kbe = valid ? (b & 0xFFFFu) : 0u;
            kbv[e] = static_cast<uint16_t>(kbe);
            if (kbe != 0u) {
                const uint32_t t = tok_of(e);
                atomicOr(&rowmask[isq ? 1 : 0][t >> 5], 1u << (t & 31u));
            }
        }
    }
    __syncthreads();   // the scratch is reused by the reverse scan

    // reverse: rex, peers after, group total; then every per-entry result
    {
        Bwd agg = {0.f, 0.f, 0u, 0.f};
#pragma unroll
        for (int k = kItems - 1; k >= 0; --k) {
            const bool tail = (tailm >> k) & 1u;
            const Bwd it = {x[k], 0.f, cnt_of(k) | ((tail ? 1u : 0u) << 31), tail ? lv[ke[k]] : 0.f};
            agg = k == kItems - 1 ? it : bcomb(agg, it);
        }
        Bwd run = bwd_block_prefix(agg, bscr, lane, warp, nw);
        zpace();
        const int64_t qbase = c * nq;
        // Unrolled by two only (the body is large; fully unrolled it spills): item k's gate and
        // entry are taken from the top of x[] / ke[], which shift up one place per iteration
        // (register moves, no local memory).
#pragma unroll 2
        for (int k = kItems - 1; k >= 0; --k) {
            const bool tail = (tailm >> k) & 1u;
            const Bwd ex = run;
            zpace();
            const float xk = x[kItems - 1];
            const uint32_t e = ke[kItems - 1];
#pragma unroll
            for (int q = kItems - 1; q > 0; --q) {
                x[q] = x[q - 1];
                ke[q] = ke[q - 1];
            }
            const Bwd it = {xk, 0.f, cnt_of(k) | ((tail ? 1u : 0u) << 31), tail ? lv[e] : 0.f};
            run = bcomb(run, it);
            if (e >= static_cast<uint32_t>(n)) continue;
            const int r = r0 + k;
            const bool valid = (validm >> k) & 1u;
            const uint32_t t = tok_of(e);
            const int j = static_cast<int>(e - t * wr);
            const bool isq = j >= W;
            const int ln = isq ? j - W : j;
            const uint32_t acnt = tail ? 0u : (ex.cnt & 0x7FFFFFFFu);
            const uint32_t after = isq ? (acnt >> 16) : (acnt & 0xFFFFu);
            const uint32_t bjv = posv[e];
            const uint32_t before = bjv & 0xFFFFu;
            const uint32_t jx = bjv >> 16;
            const uint32_t asat = min(after, kPosCountMax);
            const uint32_t pack = valid ? (static_cast<uint32_t>(r) | asat << kPosAfterShift |
                                           min(before + 1u + asat, kPosCountMax) << kPosSizeShift)
                                        : static_cast<uint32_t>(r);
            posv[e] = pack;
            const uint32_t payload = t << kTokenShift | (isq ? kIsQBit : 0u) | static_cast<uint32_t>(ln) |
                                     (valid ? 0u : kInvalidBit);
            const uint32_t el = (payload & kEntryMask) |
                                (valid ? (min(before, kDistMax) << kDistShift | (before == 0 ? kFirst : 0u) |
                                          (after == 0 ? kLast : 0u))
                                       : (kFirst | kLast));
            if (isq) {
                if (a.out.sorted_q != nullptr) st_stream(a.out.sorted_q + qbase + jx, static_cast<int32_t>(el));
            } else {
                const int o = static_cast<int>(t) * W + ln;
                const float rex = (valid && !tail) ? __fadd_rn(ex.s, ex.c) : 0.f;
                const float cpe_f = valid ? to_f(from_f<ValT>(expf(run.tot))) : 1.0f;
                rexv[o] = rex;
                cpev[o] = cpe_f;
                // the write row's word: entry | VALID | LAST | FIRST | (FIRST: the group's size,
                // else the valid write entries before it in the group) << 16
                krpos[jx] = valid ? (e | kKrValid | (after == 0 ? kKrLast : 0u) |
                                     (before == 0 ? kKrFirst | (after + 1u) << 16 : before << 16))
                                  : e;
                if (valid && before == 0)   // the group's records in its bucket: a long group has one
                    atomicAdd(&bcnt[bucket_of(keys[e])], after + 1u >= static_cast<uint32_t>(kLongMin) ? 1u : after + 1u);
                if constexpr (ORD)   // the saving forward: group heads by write-row position
                    if (valid && before == 0) atomicOr(&khead[jx >> 5], 1u << (jx & 31u));
                if (valid && before == 0 && after + 1u >= kHotMin) atomicOr(&hotmask[r >> 5], 1u << (r & 31));
            }
        }
    }
    if (a.out.repeats != nullptr) {
        const uint32_t wsum = __reduce_add_sync(kFull, repc);
        if (lane == 0 && wsum != 0u)
            atomicAdd(reinterpret_cast<unsigned long long*>(a.out.repeats), static_cast<unsigned long long>(wsum));
    }
    __syncthreads();

    // ---- DW work split: the chunk's slot groups (valid write entries) are partitioned into B
    // buckets by a hash of the slot, each group's records contiguous and in sorted order; the order
    // of groups inside a bucket does not matter (different slots). bb[p][ti][b] = the bucket's first
    // record, bb[p][ti][B] = the chunk's valid write entries (one coalesced row per chunk). Hashing spreads the hot slots of a
    // skewed stream over different DW warps.
    {
        const int B = nbk;
        uint32_t* const off = bcnt;          // [B + 1]: sizes counted by the reverse scan
        uint32_t* const fill = bcnt + B + 1; // [B]
        block_exscan_padded(off, B + 1, B + 1, uscr, lane, warp, nw);
        __syncthreads();
        zpace();
        const int64_t p = c % a.P, ti = c / a.P;
        for (int b = tid; b <= B; b += nthr) a.bb[(p * a.steps + ti) * (B + 1) + b] = static_cast<int32_t>(off[b]);
        const int64_t kbase = c * a.rstride;
        // record of the write entry with word kpi at place rec: {token | LAST | extra, slot, sc, cpe}
        auto put_record = [&](uint32_t kpi, uint32_t rec, uint32_t key, uint32_t extra) {
            const uint32_t e = kpi & kKrEntry;
            const uint32_t t = tok_of(e);
            const int o = static_cast<int>(t * W + (e - t * wr));
            const uint32_t w0 = t | ((kpi & kKrLast) ? kLast : 0u) | extra;
            const float sc = __fmul_rn(to_f(vals[e]), expf(rexv[o]));
            st_stream(a.krec + kbase + rec, make_int4(static_cast<int>(w0), static_cast<int>(key), __float_as_int(sc),
                                                      __float_as_int(cpev[o])));
        };
        // A warp takes 32 consecutive write-row positions: each writes its sorted write-row element
        // (coalesced, derived from the word); a group's first entry claims the group's place in its
        // bucket and writes the group's records (its members are the next positions of the row).
        for (int j0 = warp * 32; j0 < nk; j0 += nthr) {
            const int j = j0 + lane;
            zpace();
            uint32_t gpre = 0;   // ORD: groups before this warp's word (the dense ordinal of a group starting in it)
            if constexpr (ORD) {
                for (int wi = lane; wi < (j0 >> 5); wi += 32) gpre += __popc(khead[wi]);
                gpre = __reduce_add_sync(kFull, gpre);
            }
            const uint32_t kp = j < nk ? krpos[j] : 0u;
            if (a.out.stats != nullptr) {   // this warp's group heads
                const uint32_t hm = __ballot_sync(kFull, (kp & kKrFirst) != 0u);
                if (lane == 0 && hm != 0u) atomicAdd(&ngroups_s, static_cast<uint32_t>(__popc(hm)));
            }
            if (j < nk && a.out.sorted_k != nullptr) {
                const uint32_t e = kp & kKrEntry;
                const uint32_t t = tok_of(e);
                const uint32_t ln = e - t * wr;
                const uint32_t kb = (kp & kKrFirst) ? 0u : kp >> 16;   // valid write entries before it in the group
                st_stream(a.out.sorted_k + c * nk + j,
                          static_cast<int32_t>((kp & kKrValid)
                                                   ? (t << kTokenShift | ln | min(kb, kDistMax) << kDistShift |
                                                      ((kp & kKrFirst) ? kFirst : 0u) | ((kp & kKrLast) ? kLast : 0u))
                                                   : ((t << kTokenShift | ln | kInvalidBit) | kFirst | kLast)));
            }
            if (kp & kKrFirst) {
                const uint32_t e = kp & kKrEntry;
                const uint32_t key = keys[e];
                const uint32_t b = bucket_of(key);
                const uint32_t size = kp >> 16;
                if (size >= static_cast<uint32_t>(kLongMin)) {
                    // long: its reference record in the bucket {index | kRecLong | FIRST | LAST (| ordinal),
                    // slot, row of the sums, cpe}; its own records in the chunk's tail (below)
                    const uint32_t li = atomicAdd(&lcnt_s, 1u);   // < C*W / kLongMin
                    const uint32_t ref = off[b] + atomicAdd(&fill[b], 1u);
                    const uint32_t base = off[B] + atomicAdd(&ltail_s, size);
                    a.ldesc[c * a.maxL + li] = static_cast<int32_t>(base);
                    const uint32_t t = tok_of(e);
                    uint32_t w0 = li | kRecLong | kFirst | kLast;
                    if constexpr (ORD) {   // the group's dense ordinal (khead is complete: reverse scan)
                        uint32_t g = __popc(khead[j >> 5] & ((1u << (j & 31)) - 1u));
                        for (int wi = 0; wi < (j >> 5); ++wi) g += __popc(khead[wi]);
                        w0 |= g << kRecOrdShift;
                    }
                    st_stream(a.krec + kbase + ref,
                              make_int4(static_cast<int>(w0), static_cast<int>(key), static_cast<int>(c * a.maxL + li),
                                        __float_as_int(cpev[static_cast<int>(t) * W + static_cast<int>(e - t * wr)])));
                    krpos[j] = (kp & 0xFFFFu) | base << 16 | kKrLong;   // the group's first tail record
                } else {
                    const uint32_t base = off[b] + atomicAdd(&fill[b], size);
                    uint32_t first = kFirst;
                    if constexpr (ORD)   // the group's dense ordinal
                        first |= (gpre + __popc(khead[j0 >> 5] & ((1u << lane) - 1u))) << kRecOrdShift;
                    put_record(kp, base, key, first);
                    for (uint32_t q = 1; q < size; ++q) put_record(krpos[j + q], base + q, key, 0u);
                }
            }
        }
        __syncthreads();
        if constexpr (ORD) {
            if (warp == 0 && a.out.ngroups != nullptr) {   // the chunk's valid write groups
                const int nwords = (nk + 31) >> 5;
                uint32_t cnt = 0;
                for (int wi = lane; wi < nwords; wi += 32) cnt += __popc(khead[wi]);
                cnt = __reduce_add_sync(kFull, cnt);
                if (lane == 0) a.out.ngroups[c] = static_cast<int32_t>(cnt);
            }
        }
        if (lcnt_s != 0u) {   // long groups: every member writes its own record in the chunk's tail
            for (int j0 = warp * 32; j0 < nk; j0 += nthr) {
                uint32_t gpre = 0;
                if constexpr (ORD) {
                    for (int wi = lane; wi < (j0 >> 5); wi += 32) gpre += __popc(khead[wi]);
                    gpre = __reduce_add_sync(kFull, gpre);
                }
                const int j = j0 + lane;
                if (j >= nk) continue;
                const uint32_t kp = krpos[j];
                if (!(kp & kKrValid)) continue;
                const uint32_t kb = (kp & kKrFirst) ? 0u : kp >> 16;
                const uint32_t f = krpos[j - kb];
                if (!(f & kKrLong)) continue;
                uint32_t first = 0u;
                if (kb == 0u) {
                    first = kFirst;
                    if constexpr (ORD) first |= (gpre + __popc(khead[j0 >> 5] & ((1u << lane) - 1u))) << kRecOrdShift;
                }
                put_record(kp, ((f & ~kKrLong) >> 16) + kb, keys[kp & kKrEntry], first);
            }
        }
    }

    // ---- 3. entry-order outputs -------------------------------------------------------------------
    {
        zpace();
        const int64_t kbase = c * nk;
        ValT* const cpe_o = static_cast<ValT*>(a.out.cpe);
        ValT* const keff_o = static_cast<ValT*>(a.out.k_eff);
        const int64_t qbase = c * nq;
        ValT* const qw_o = static_cast<ValT*>(a.out.q_w);
        if ((W & 3) == 0 && (R & 3) == 0) {
            // four consecutive entries of one token per thread: vector loads from shared memory
            // (their entry indices are consecutive and a multiple of 4) and vector stores
            for (int o = 4 * tid; o < nk; o += 4 * nthr) {
                const int t = static_cast<int>(__umulhi(static_cast<uint32_t>(o), a.w_magic)), e = t * wr + (o - t * W);
                zpace();
                const uint4 pk = *reinterpret_cast<const uint4*>(posv + e);
                float lg[4], v[4];
                ld4(lv + e, lg);
                const uint32_t p4[4] = {pk.x, pk.y, pk.z, pk.w};
                if (a.out.log_k) st4(a.out.log_k + kbase + o, lg);
                if (a.out.rex) {
                    float r4[4];
                    ld4(rexv + o, r4);
                    st4(a.out.rex + kbase + o, r4);
                }
                if (cpe_o) {
                    float c4[4];
                    ld4(cpev + o, c4);
                    st4(cpe_o + kbase + o, c4);
                }
                if (keff_o) {
                    ld4(vals + e, v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = ((p4[q] >> kPosSizeShift) & kPosCountMax) != 0u ? v[q] * expf(lg[q]) : 0.f;
                    st4(keff_o + kbase + o, v);
                }
                auto last = [&](int q) -> uint32_t {
                    return ((p4[q] >> kPosSizeShift) & kPosCountMax) != 0u && ((p4[q] >> kPosAfterShift) & kPosCountMax) == 0u;
                };
                auto only = [&](int q) -> uint32_t { return ((p4[q] >> kPosSizeShift) & kPosCountMax) == 1u; };
                if (a.out.is_last) st4_flags(a.out.is_last + kbase + o, last(0), last(1), last(2), last(3));
                if (a.out.is_only) st4_flags(a.out.is_only + kbase + o, only(0), only(1), only(2), only(3));
                if (a.out.pos_k) st_na(reinterpret_cast<uint4*>(a.out.pos_k + kbase + o), pk);
            }
            for (int o = 4 * tid; o < nq; o += 4 * nthr) {
                const int t = static_cast<int>(__umulhi(static_cast<uint32_t>(o), a.r_magic)), e = t * wr + W + (o - t * R);
                zpace();
                const uint4 pk = *reinterpret_cast<const uint4*>(posv + e);
                float lg[4], v[4];
                ld4(lv + e, lg);
                const uint32_t p4[4] = {pk.x, pk.y, pk.z, pk.w};
                if (a.out.log_q) st4(a.out.log_q + qbase + o, lg);
                if (qw_o) {
                    ld4(vals + e, v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = ((p4[q] >> kPosSizeShift) & kPosCountMax) != 0u ? v[q] * expf(lg[q]) : 0.f;
                    st4(qw_o + qbase + o, v);
                }
                auto last = [&](int q) -> uint32_t {
                    return ((p4[q] >> kPosSizeShift) & kPosCountMax) != 0u && ((p4[q] >> kPosAfterShift) & kPosCountMax) == 0u;
                };
                auto only = [&](int q) -> uint32_t { return ((p4[q] >> kPosSizeShift) & kPosCountMax) == 1u; };
                if (a.out.q_last) st4_flags(a.out.q_last + qbase + o, last(0), last(1), last(2), last(3));
                if (a.out.q_only) st4_flags(a.out.q_only + qbase + o, only(0), only(1), only(2), only(3));
                if (a.out.pos_q) st_na(reinterpret_cast<uint4*>(a.out.pos_q + qbase + o), pk);
            }
        } else {
            for (int o = tid; o < nk; o += nthr) {
                const int t = static_cast<int>(__umulhi(static_cast<uint32_t>(o), a.w_magic)), e = t * wr + (o - t * W);
                const uint32_t pk = posv[e];
                const uint32_t size = (pk >> kPosSizeShift) & kPosCountMax;
                const bool valid = size != 0u;
                const float lg = lv[e];
                if (a.out.log_k) st_stream(a.out.log_k + kbase + o, lg);
                if (a.out.rex) st_stream(a.out.rex + kbase + o, rexv[o]);
                if (cpe_o) st_stream(cpe_o + kbase + o, from_f<ValT>(cpev[o]));
                if (keff_o) st_stream(keff_o + kbase + o, from_f<ValT>(valid ? to_f(vals[e]) * expf(lg) : 0.f));
                if (a.out.is_last)
                    st_stream(a.out.is_last + kbase + o, static_cast<int8_t>(valid && ((pk >> kPosAfterShift) & kPosCountMax) == 0u));
                if (a.out.is_only) st_stream(a.out.is_only + kbase + o, static_cast<int8_t>(size == 1u));
                if (a.out.pos_k) st_stream(a.out.pos_k + kbase + o, static_cast<int32_t>(pk));
            }
            for (int o = tid; o < nq; o += nthr) {
                const int t = static_cast<int>(__umulhi(static_cast<uint32_t>(o), a.r_magic)), e = t * wr + W + (o - t * R);
                const uint32_t pk = posv[e];
                const uint32_t size = (pk >> kPosSizeShift) & kPosCountMax;
                const bool valid = size != 0u;
                const float lg = lv[e];
                if (a.out.log_q) st_stream(a.out.log_q + qbase + o, lg);
                if (qw_o) st_stream(qw_o + qbase + o, from_f<ValT>(valid ? to_f(vals[e]) * expf(lg) : 0.f));
                if (a.out.q_last)
                    st_stream(a.out.q_last + qbase + o, static_cast<int8_t>(valid && ((pk >> kPosAfterShift) & kPosCountMax) == 0u));
                if (a.out.q_only) st_stream(a.out.q_only + qbase + o, static_cast<int8_t>(size == 1u));
                if (a.out.pos_q) st_stream(a.out.pos_q + qbase + o, static_cast<int32_t>(pk));
            }
        }
    }

    // ---- 4. pair triangles --------------------------------------------------------------------------
    if (tid == 0) a.lcnt[c] = static_cast<int32_t>(lcnt_s);   // final since the DW split's barrier
    if (tid == 0 && a.out.stats != nullptr && ngroups_s != 0u)
        atomicAdd(reinterpret_cast<unsigned long long*>(a.out.stats), static_cast<unsigned long long>(ngroups_s));
    if (a.out.A == nullptr && a.out.QK == nullptr) return;
    while (zero_next < zka + zkq) zero_store();   // the units left; the barrier orders them before the rows' stores
    __syncthreads();   // the key array becomes the row buffers
    float* const rowbuf = reinterpret_cast<float*>(smem + a.sm_keys) + warp * C;
    const uint32_t le = lanemask_le();
    const bool vec4 = (C % 4) == 0;

    // Dense path of hot slot groups. Inside a group the entries run in token order, every write
    // entry of token j before every entry of token i > j and, within a token, its write entries
    // before its read entries. So the group adds to A[i][j] (j < i) and QK[i][j] (j <= i)
    //   sum_a sum_b v_a v_b exp(L_a - L_b) = UK[i] * WK[j]   (QK: UQ[i] * WK[j]),
    //   UK[i] = sum over token i's write entries a of v_a exp(L_a - ref), UQ the same over its
    //   read entries, WK[j] = sum over token j's write entries b of v_b exp(ref - L_b),
    // a rank-1 term per group. ref = L_first - 40 keeps both factors within e^{+-40} when the
    // group's log-cumsums span at most kHotSpan; a wider group keeps the exact walk. The first
    // (in position order) groups with at least kHotMin write entries take this path, as many as
    // the free shared memory holds; their entries are marked (kb bit 15) and skip the walk.
    struct HotMeta {
        int r0, r1, ok;
        float ref;
    };
    static_assert(sizeof(HotMeta) == 16, "the host sizes the dense path's region with 16-byte descriptors");
    HotMeta* const meta = reinterpret_cast<HotMeta*>(smem + a.sm_rex);   // rex .. zero buffer: free now
    float* const hvec = reinterpret_cast<float*>(smem + a.sm_rex + kHotMax * sizeof(HotMeta));
    const int hot_cap = a.hot_cap;   // from the shape alone: the same groups go dense for any geometry
    if (warp == 0) {   // the first hot_cap candidates in position order
        const int nwords = npad >> 5;
        uint32_t cnt = 0;
        for (int q = 0; q < 8; ++q) {
            const int wi = lane * 8 + q;
            if (wi < nwords) cnt += __popc(hotmask[wi]);
        }
        uint32_t incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += y;
        }
        int idx = static_cast<int>(incl - cnt);
        for (int q = 0; q < 8 && idx < hot_cap; ++q) {
            const int wi = lane * 8 + q;
            for (uint32_t m = wi < nwords ? hotmask[wi] : 0u; m != 0u && idx < hot_cap; m &= m - 1u)
                meta[idx++].r0 = wi * 32 + __ffs(m) - 1;
        }
        if (lane == 31) hot_n = min(static_cast<int>(incl), hot_cap);
    }
    __syncthreads();
    const int nhot = hot_n;
    for (int h = warp; h < nhot; h += nw) {   // one warp builds a group's vectors
        const int hr0 = meta[h].r0;
        const uint32_t hkey = keys[sidx[hr0]];
        const float l0 = lv[sidx[hr0]];
        int hr1 = hr0;   // the group's last position: same key
        for (int base = hr0 + 1;; base += 32) {
            const int pos = base + lane;
            const uint32_t m = __ballot_sync(kFull, pos < npad && keys[sidx[pos]] == hkey);
            if (m != kFull) {
                hr1 = base + __ffs(~m) - 2;
                break;
            }
        }
        const bool ok = __fsub_rn(l0, lv[sidx[hr1]]) <= kHotSpan;
        const float ref = __fsub_rn(l0, 40.f);
        if (lane == 0) {
            meta[h].r1 = hr1;
            meta[h].ok = ok ? 1 : 0;
            meta[h].ref = ref;
        }
        if (!ok) continue;
        float* const uk = hvec + h * 3 * C;
        float* const uq = uk + C;
        float* const wk = uq + C;
        for (int j = lane; j < 3 * C; j += 32) uk[j] = 0.f;
        __syncwarp();
        for (int base = hr0; base <= hr1; base += 32) {
            const int pos = base + lane;
            float vk = 0.f, vq = 0.f, vw = 0.f;
            int tf = -1;
            if (pos <= hr1) {
                const uint32_t f = sidx[pos];
                tf = static_cast<int>(tok_of(f));
                const float vf = to_f(vals[f]), lf = lv[f];
                const float u = __fmul_rn(vf, expf(__fsub_rn(lf, ref)));
                if (is_q_of(f)) {
                    vq = u;
                } else {
                    vk = u;
                    vw = __fmul_rn(vf, expf(__fsub_rn(ref, lf)));
                }
                kbv[f] = static_cast<uint16_t>(kbv[f] | 0x8000u);   // handled densely
            }
            // per-token sums over the lanes (tokens are non-decreasing along the lanes): a fixed
            // shuffle tree, the token's first lane adds them to the vectors
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float ok_ = __shfl_down_sync(kFull, vk, d);
                const float oq = __shfl_down_sync(kFull, vq, d);
                const float ow = __shfl_down_sync(kFull, vw, d);
                const int ot = __shfl_down_sync(kFull, tf, d);
                if (lane + d < 32 && ot == tf) {
                    vk = __fadd_rn(vk, ok_);
                    vq = __fadd_rn(vq, oq);
                    vw = __fadd_rn(vw, ow);
                }
            }
            const int tprev = __shfl_up_sync(kFull, tf, 1);
            if (tf >= 0 && (lane == 0 || tprev != tf)) {
                uk[tf] = __fadd_rn(uk[tf], vk);
                uq[tf] = __fadd_rn(uq[tf], vq);
                wk[tf] = __fadd_rn(wk[tf], vw);
                const uint32_t hb = 1u << h;   // kHotMax <= 32
                if (vk != 0.f) atomicOr(&hotrow[0][tf], hb);
                if (vq != 0.f) atomicOr(&hotrow[1][tf], hb);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    if (tid == 0 && a.out.stats != nullptr && nhot > 0) {   // the groups that took the dense path
        uint32_t nd = 0;
        for (int h = 0; h < nhot; ++h) nd += meta[h].ok ? 1u : 0u;
        if (nd != 0u) atomicAdd(reinterpret_cast<unsigned long long*>(a.out.stats) + 1, static_cast<unsigned long long>(nd));
    }
    // Only rows flagged in the scan (an entry with an earlier write entry in its group) have
    // terms. Lane u < 2 * mwords holds flag word u (A rows, then QK rows); a warp prefix of the
    // words' counts locates the j-th flagged (triangle, row) pair without any walk over the others.
    const int mwords = (C + 31) >> 5;   // <= 8: the flag words fit the lanes
    const uint32_t fw = lane < 2 * mwords ? rowmask[lane >= mwords ? 1 : 0][lane >= mwords ? lane - mwords : lane] : 0u;
    uint32_t fincl = __popc(fw);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, fincl, d);
        if (lane >= d) fincl += y;
    }
    const uint32_t fexcl = fincl - __popc(fw);
    const uint32_t nflag = __shfl_sync(kFull, fincl, 31);
    // warps take the flagged pairs from a counter (rows differ in work: skewed chunks balance)
    uint32_t nterm = 0, nrow = 0;   // out.stats: exact pair terms and rows written by this warp
    for (;;) {
        uint32_t jf = 0;
        if (lane == 0) jf = atomicAdd(&row_claim, 1u);
        jf = __shfl_sync(kFull, jf, 0);
        if (jf >= nflag) break;
        const int u = __ffs(__ballot_sync(kFull, jf >= fexcl && jf < fincl)) - 1;   // the word holding pair jf
        uint32_t bits = __shfl_sync(kFull, fw, u);
        for (uint32_t q = __shfl_sync(kFull, fexcl, u); q < jf; ++q) bits &= bits - 1u;
        const bool qk = u >= mwords;
        float* const outp = qk ? a.out.QK : a.out.A;
        if (outp == nullptr) continue;
        const int i = (qk ? u - mwords : u) * 32 + __ffs(bits) - 1;
        bool any = false;
        const int lanes = qk ? R : W;
        for (int ab0 = 0; ab0 < lanes; ab0 += 32) {
            // the row's entries with an earlier write entry in their group, one ballot per 32
            const int eab = i * wr + (qk ? W : 0) + ab0 + lane;
            uint32_t with = __ballot_sync(kFull, ab0 + lane < lanes && static_cast<uint32_t>(kbv[eab]) - 1u < 0x7FFFu);
            for (; with != 0u; with &= with - 1u) {
                const int e = i * wr + (qk ? W : 0) + ab0 + __ffs(with) - 1;
                const uint32_t kb = kbv[e];
                if (!any) {
                    for (int j = lane; j < C; j += 32) rowbuf[j] = 0.f;
                    __syncwarp();
                    any = true;
                }
                const int r = static_cast<int>(posv[e] & kPosMask);
                const float ve = to_f(vals[e]), lge = lv[e];
                uint32_t met = 0;
                for (int top = r - 1; met < kb && top >= 0; top -= 32) {
                    const int p = top - lane;
                    const bool in = p >= 0;
                    uint32_t f = 0;
                    bool isk = false;
                    if (in) {
                        f = sidx[p];
                        isk = f < static_cast<uint32_t>(n) && !is_q_of(f) &&
                              ((posv[f] >> kPosSizeShift) & kPosCountMax) != 0u;
                    }
                    const uint32_t bk = __ballot_sync(kFull, isk);
                    const uint32_t before_me = __popc(bk & le) - (isk ? 1u : 0u);
                    const bool incl = in && (met + before_me < kb);
                    const int tf = incl ? static_cast<int>(tok_of(f)) : -1;
                    float v = 0.f;
                    if (a.out.stats != nullptr) nterm += __popc(__ballot_sync(kFull, incl && isk && (qk || tf != i)));
                    if (incl && isk && (qk || tf != i)) {
                        v = __fmul_rn(__fmul_rn(ve, to_f(vals[f])), expf(__fsub_rn(lge, lv[f])));
                    }
                    const uint32_t terms = __ballot_sync(kFull, v != 0.f);
                    if ((terms & (terms - 1u)) == 0u) {   // at most one term: it is the cell's sum
                        if (v != 0.f) rowbuf[tf] = __fadd_rn(rowbuf[tf], v);
                    } else {
                        // segmented suffix sums over lanes of equal token (tokens are non-increasing
                        // along the lanes): a fixed shuffle tree
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {
                            const float ov = __shfl_down_sync(kFull, v, d);
                            const int ot = __shfl_down_sync(kFull, tf, d);
                            if (lane + d < 32 && ot == tf) v = __fadd_rn(v, ov);
                        }
                        const int tprev = __shfl_up_sync(kFull, tf, 1);
                        if (tf >= 0 && (lane == 0 || tprev != tf)) rowbuf[tf] = __fadd_rn(rowbuf[tf], v);
                    }
                    __syncwarp();
                    met += __popc(bk);
                }
            }
        }
        // the rank-1 terms of the dense groups with an entry of this token, in group order, added
        // to the row held in registers (column lane + 32 q)
        uint32_t hm = hotrow[qk ? 1 : 0][i];
        if (hm != 0u) {
            __syncwarp();
            float racc[kMaxC / 32];
#pragma unroll
            for (int q = 0; q < kMaxC / 32; ++q) {
                const int j = lane + 32 * q;
                racc[q] = (any && j < C) ? rowbuf[j] : 0.f;
            }
            const int jend = qk ? i + 1 : i;   // columns j < jend
            for (; hm != 0u; hm &= hm - 1u) {
                const float* const uk = hvec + (__ffs(hm) - 1) * 3 * C;
                const float coef = qk ? uk[C + i] : uk[i];
#pragma unroll
                for (int q = 0; q < kMaxC / 32; ++q) {
                    const int j = lane + 32 * q;
                    if (j < jend) racc[q] = fmaf(coef, uk[2 * C + j], racc[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < kMaxC / 32; ++q) {
                const int j = lane + 32 * q;
                if (j < C) rowbuf[j] = racc[q];
            }
            any = true;
        }
        __syncwarp();
        if (!any) continue;   // the row stays as the zero fill left it
        ++nrow;
        float* const row = outp + (c * C + i) * static_cast<int64_t>(C);
        if (vec4) {
            for (int j = lane * 4; j < C; j += 128)
                st_na(reinterpret_cast<float4*>(row + j), *reinterpret_cast<const float4*>(rowbuf + j));
        } else {
            for (int j = lane; j < C; j += 32) st_na(row + j, rowbuf[j]);
        }
        __syncwarp();
    }
    if (a.out.stats != nullptr && lane == 0) {
        unsigned long long* const st = reinterpret_cast<unsigned long long*>(a.out.stats);
        if (nterm != 0u) atomicAdd(st + 2, static_cast<unsigned long long>(nterm));
        if (nrow != 0u) atomicAdd(st + 3, static_cast<unsigned long long>(nrow));
    }
}

}  // namespace

template <typename ValT, bool ORD>
cudaError_t launch_p1(const P1Args& a, int64_t nchunks, int threads, size_t smem, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(p1_kernel<ValT, ORD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    p1_kernel<ValT, ORD><<<dim3(static_cast<unsigned>(nchunks)), threads, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_phase1(const P1Args& a, int val_bf16, int ordinals, int64_t nchunks, int threads, size_t smem,
                          cudaStream_t stream) {
    if (nchunks <= 0) return cudaSuccess;
    if (val_bf16)
        return ordinals ? launch_p1<__nv_bfloat16, true>(a, nchunks, threads, smem, stream)
                        : launch_p1<__nv_bfloat16, false>(a, nchunks, threads, smem, stream);
    return ordinals ? launch_p1<float, true>(a, nchunks, threads, smem, stream)
                    : launch_p1<float, false>(a, nchunks, threads, smem, stream);
}

cudaError_t phase1_smem_limit(int device, size_t* bytes) {
    int v = 0;
    cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    *bytes = static_cast<size_t>(v);
    return cudaSuccess;
}

}  // namespace sdm
