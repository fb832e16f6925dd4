// sdm_internal.cuh -- shared definitions of the sm_103a kernels behind include/sdm.h.
//
// Bit layouts follow sparse-delta-memory 2.0.0 (phase1_cuda.py, p1_scan_kernel and the
// Records comment): the payload / sorted-row entry bits (lane | isQ << 8 | token << 9 |
// invalid << 17), FIRST = bit 31, LAST = bit 30, distance-to-FIRST at bits 18..29, and the
// position pack (r | after << 17 | size << 24, counts saturating at 127).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

#include "../../include/sdm.h"

namespace sdm {

// ---- layouts fixed by the method --------------------------------------------------------------
constexpr uint32_t kIsQBit = 1u << 8;
constexpr int kTokenShift = 9;
constexpr uint32_t kInvalidBit = 1u << 17;
constexpr uint32_t kEntryMask = 0x3FFFFu;
constexpr uint32_t kFirst = 1u << 31;
constexpr uint32_t kLast = 1u << 30;
constexpr int kDistShift = 18;
constexpr uint32_t kDistMax = 4095u;
constexpr int kPosBits = 17;
constexpr uint32_t kPosMask = (1u << kPosBits) - 1u;
constexpr int kPosAfterShift = 17;
constexpr int kPosSizeShift = 24;
constexpr uint32_t kPosCountMax = 127u;

// ---- this implementation's limits and geometry ------------------------------------------------
constexpr int kMaxC = 256;
constexpr int kMaxLanes = 256;          // W, R (8-bit lane field)
constexpr int kItems = 8;               // sorted positions per thread in the Phase-1 kernel
constexpr int kMaxThreads = 1024;
constexpr int kMaxRow = kItems * kMaxThreads;   // entries of one chunk held on chip
constexpr uint32_t kKeyInvalid = 1u << 31;       // key word flag: not a valid entry
constexpr int kSortDigitBits = 4;               // radix digit of the Phase-1 sort
constexpr int kSortDigits = 1 << kSortDigitBits;
// a sort word between passes: the entry in the low kSortWordEntryBits bits (kMaxRow entries), the
// key bits still to sort above it once they fit
constexpr int kSortWordEntryBits = 13;
constexpr uint32_t kSortWordEntryMask = (1u << kSortWordEntryBits) - 1u;
constexpr int kSortWordKeyBits = 32 - kSortWordEntryBits;
static_assert(kMaxRow <= (1 << kSortWordEntryBits), "a sort word holds an entry index");
// Phase 1's word per write-row position: the entry (13 bits), LAST, FIRST, VALID and, from bit
// 16, the group's size (FIRST; later the group's first record) or the valid write entries before
// the entry in its group
constexpr uint32_t kKrEntry = 0x1FFFu;
constexpr uint32_t kKrLast = 1u << 13;
constexpr uint32_t kKrFirst = 1u << 14;
constexpr uint32_t kKrValid = 1u << 15;
// set by the DW split in a long group's FIRST word, whose bits 16..30 then hold the group's first
// record in the chunk's tail
constexpr uint32_t kKrLong = 1u << 31;
// the Phase-1 sort's fast path: a counting sort by the key's top kBucketBits bits (buckets of 32-bit
// counts in the position-pack region), taken when no bucket holds more than kBucketMax entries
constexpr int kBucketBits = 13;
constexpr int kBucketMax = 16;
// Phase 1: SM clock cycles between a warp's zero stores of A / QK (one 16-byte unit per thread)
constexpr uint32_t kZeroPeriod = 1400u;
// bytes of the Phase-1 shared memory after the bucket counters, part of the dense pair path's room
constexpr int kHotExtra = 4096;
// bound on the Phase-1 kernel's static shared memory (its flag words and counters)
constexpr size_t kP1StaticSmem = 6144;
// dense pair path: slot groups with at least kHotMin write entries, at most kHotMax per chunk,
// whose log-cumsums span at most kHotSpan
constexpr uint32_t kHotMin = 16;
constexpr int kHotMax = 16;
constexpr float kHotSpan = 80.f;
constexpr size_t kSmemOptin = 232448;          // opt-in shared memory per block on sm_103a

// Device status word bits (mirrors SDM_DEV_* in sdm.h).
constexpr uint32_t kDevBadSlot = SDM_DEV_BAD_SLOT;

// DW record of one valid write entry (16 bytes, one vector load), grouped by slot bucket:
//   x = token | group ordinal << 16 (FIRST records) | kRecLong | LAST << 30 | FIRST << 31,
//   y = stream-local slot,
//   z = f32 bits of sc = k * expf(rex), w = f32 bits of cpe (the value-type cpe widened).
constexpr uint32_t kRecTokMask = 0xFFFFu;
// A long group (at least kLongMin write entries in its chunk, e.g. a hot slot of a skewed stream)
// takes ONE record in its slot bucket -- the reference record: x = the group's index among the
// chunk's long groups | kRecLong | FIRST | LAST (| ordinal), y = slot, z = its row of the sums
// (chunk * maxL + index), w = cpe -- while its own
// records go to the chunk's tail (after the buckets' records), where the long-group kernel sums
// them (the DW walk's very FMA chain) before the DW, which takes the sum at the reference record.
constexpr uint32_t kRecLong = 1u << 29;
constexpr int kLongMin = 8;
constexpr int kMaxLong = kMaxRow / kLongMin;   // long groups per chunk at most
static_assert(kMaxRow + kMaxLong < (1 << 15), "a chunk's record places fit bits 16..30 of a write-row word");
// the group's dense ordinal in its chunk (valid write groups before it in sorted order), carried by
// the group's FIRST record: the row of the dense compact snapshot
constexpr int kRecOrdShift = 16;
constexpr uint32_t kRecOrdMask = 0x1FFFu;

// Workspace header (bytes): [0] status word, [4] the DW work counter.
constexpr size_t kHdrStatus = 0;
constexpr size_t kHdrClaim = 4;
constexpr size_t kHdrBytes = 256;

struct Geometry {
    int C, W, R, wr, n, nk, nq, P, hd;
    int64_t steps, N, S;
    int key_bits, passes, digit_bits;
    int bucket_bits;       // min(key_bits, kBucketBits, floor(log2(npad)))
    int threads, npad, nwarps;
    int B, logB;           // DW buckets per stream, B = 2^logB: a slot group's bucket is a hash of its slot
    int nsl;               // DW column slices of 128 columns
    size_t krec_off, bb_off, lcnt_off, ldesc_off, lacc_off, ws_bytes;
    int maxL;              // long groups per chunk at most: max(1, C*W / kLongMin)
    int rstride;           // records per chunk: C*W + maxL (a long group adds its reference record)
    size_t smem_bytes;
    int hot_cap;           // dense pair groups per chunk at most (from the shape alone)
    // Phase-1 shared-memory carve (byte offsets)
    size_t sm_keys, sm_vals, sm_sidx, sm_regd, sm_pong, sm_hist, sm_pos, sm_kb, sm_rex, sm_tot, sm_kslot, sm_bcnt,
        sm_zero, sm_scr;
};

struct P1Args {
    const int32_t* k_idx;
    const int32_t* q_idx;
    const void* k_val;
    const void* q_val;
    const float* g;
    sdm_p1_out out;
    int4* krec;
    int32_t* bb;            // [P][steps][B + 1] first record of each slot bucket, per chunk
    int32_t* lcnt;          // [N] long groups of each chunk
    int32_t* ldesc;         // [N][maxL] the first tail record of each long group
    int maxL, rstride;
    uint32_t* status;
    int C, W, R, wr, n, nk, nq, npad, nwarps;
    int key_bits, passes, digit_bits;
    int bucket_bits;        // the sort's fast path: buckets of the key's top bucket_bits bits
    int64_t S;
    int64_t c0;             // first chunk of the launch
    int64_t first_partial;  // first chunk whose tokens t >= valid_last are invalid
    int valid_last;
    int g_width, g_lane_stride;
    uint32_t wr_magic;      // ceil(2^32 / wr): e / wr == umulhi(e, wr_magic) for e * wr < 2^32
    uint32_t w_magic, r_magic;   // the same for W and R (entry-order output index -> token)
    int P, logB;
    int64_t steps;
    int hot_cap;            // dense pair groups per chunk at most
    uint32_t sm_keys, sm_vals, sm_sidx, sm_pong, sm_hist, sm_pos, sm_kb, sm_rex, sm_tot, sm_kslot, sm_bcnt, sm_zero,
        sm_scr, sm_lv;
};

struct DWArgs {
    const int4* krec;
    const int32_t* bb;  // [P][steps][B + 1]
    const void* dv;
    void* bank;
    void* snap;         // dense compact snapshot [N, C*W, hd] (bank type) or null
    const float* lacc;  // [N][maxL][hd] each long group's sum of terms
    uint32_t* claim;    // work counter
    int P, C, W, nk, B, nsl, hd, maxL, rstride;
    int64_t S, steps;
    int64_t step_begin, step_end;
    int64_t items;      // P * B * nsl
};

// A launch as a programmatic dependent of the previous kernel in the stream: its CTAs may be
// scheduled before that kernel completes (onto SMs it leaves idle) and wait in the kernel
// (griddepcontrol.wait) until it has completed and its memory is visible. Every kernel launched so
// waits before its first memory access, so stream order holds whatever kernel came before.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_phase1(const P1Args& a, int val_bf16, int ordinals, int64_t nchunks, int threads, size_t smem,
                          cudaStream_t stream);
cudaError_t launch_dw(const DWArgs& a, int dv_bf16, int bank_bf16, cudaStream_t stream);
// the long groups' sums of terms, for the chunks [c0, c0 + nchunks)
struct LongArgs {
    const int4* krec;
    const int32_t* lcnt;
    const int32_t* ldesc;
    const void* dv;
    float* lacc;
    uint32_t* claim;    // the DW's work counter, zeroed here (the DW launch follows this one)
    int C, maxL, rstride, hd, nsl;
    int64_t c0, nchunks;
};
cudaError_t launch_long(const LongArgs& a, int dv_bf16, cudaStream_t stream);
cudaError_t phase1_smem_limit(int device, size_t* bytes);

}  // namespace sdm
