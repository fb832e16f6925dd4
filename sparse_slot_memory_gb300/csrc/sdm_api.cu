// sdm_api.cu -- the extern "C" entry points declared in include/sdm.h: argument checks, the
// workspace layout and the launches. Every check runs before any launch; nothing here allocates.
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

 // DW work items (stream, slot bucket, column slice) aimed at per launch: ~3x the warps a GB300 holds.
constexpr int64_t kDwTargetItems = 32768;
constexpr int kMaxLogBuckets = 11;   // the most a caller may ask for (sdm_shape.dw_log_buckets)
// The most chosen by default. Each bucket costs Phase 1 8 bytes of shared memory per CTA: with 2^11
// buckets a 512-thread CTA (C * (W + R) = 4096) needed 120 KB, one CTA per SM; with 2^10 it needs
// 112 KB and two CTAs share an SM (zipf_c256: Phase 1 455 -> 326 us; its DW and that of
// uniform_c128 are faster too with the fewer, fuller buckets).
constexpr int kAutoLogBuckets = 10;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Derives every size and offset from the shape alone. Returns SDM_OK or the error code.
sdm_status geometry(const sdm_shape* s, Geometry* g) {
    if (s == nullptr) return SDM_ERR_ARG;
    if (s->val_dtype < 0 || s->val_dtype > 1 || s->dv_dtype < 0 || s->dv_dtype > 1 || s->bank_dtype < 0 ||
        s->bank_dtype > 1)
        return SDM_ERR_DTYPE;
    if (s->P < 1 || s->C < 1 || s->C > kMaxC || s->W < 1 || s->W > kMaxLanes || s->R < 1 || s->R > kMaxLanes ||
        s->steps < 1 || s->S < 1 || s->S > 0x7FFFFFFFll || s->hd < 1 || s->valid_last < 1 || s->valid_last > s->C ||
        (s->gate_per_entry != 0 && s->gate_per_entry != 1))
        return SDM_ERR_SHAPE;
    if (s->hd % 4 != 0) return SDM_ERR_ALIGN;
    const int64_t n = static_cast<int64_t>(s->C) * (s->W + s->R);
    if (n > kMaxRow) return SDM_ERR_SHAPE;
    if (s->steps > (int64_t(1) << 40) / s->P) return SDM_ERR_SHAPE;
    const int64_t N = s->steps * s->P;
    // every flattened index must fit int64 with room: bank rows, dv rows, A/QK cells
    if (s->S > (int64_t(1) << 62) / s->P / s->hd) return SDM_ERR_SHAPE;
    if (N > (int64_t(1) << 62) / (static_cast<int64_t>(s->C) * s->C + s->C * int64_t(s->hd) + n)) return SDM_ERR_SHAPE;
    memset(g, 0, sizeof(*g));
    g->C = s->C;
    g->W = s->W;
    g->R = s->R;
    g->wr = s->W + s->R;
    g->n = static_cast<int>(n);
    g->nk = s->C * s->W;
    g->nq = s->C * s->R;
    g->P = s->P;
    g->hd = s->hd;
    g->steps = s->steps;
    g->N = N;
    g->S = s->S;
    int kb = 1;
    while ((int64_t(1) << kb) < s->S) ++kb;
    g->key_bits = kb;
    g->passes = (kb + kSortDigitBits - 1) / kSortDigitBits;
    g->digit_bits = kSortDigitBits;
    int threads = static_cast<int>((n + kItems - 1) / kItems);
    threads = static_cast<int>(round_up(static_cast<size_t>(threads), 32));
    if (s->p1_warps != 0) {   // a wider block: the extra warps hold padding entries
        if (s->p1_warps < threads / 32 || s->p1_warps > kMaxThreads / 32) return SDM_ERR_SHAPE;
        threads = s->p1_warps * 32;
    }
    g->threads = threads;
    g->npad = threads * kItems;
    g->nwarps = threads / 32;
    {   // the sort's bucket counts (uint32) lie in the position-pack region of npad words
        int lg = 0;
        while ((2 << lg) <= g->npad) ++lg;
        g->bucket_bits = std::min(std::min(kb, kBucketBits), lg);
    }
    g->nsl = (s->hd + 127) / 128;
    // DW buckets per stream: about kDwTargetItems / nsl items per launch (a row of nsl 128-column
    // slices is walked by nsl items that each read all of the bucket's records: wide rows want fuller
    // buckets; hd = 960 measured 130 -> 119 us with 128 instead of 1024 buckets per stream, 163 us
    // with 64), at most 2^kAutoLogBuckets and no more buckets than 2^key_bits
    int64_t want = kDwTargetItems / (static_cast<int64_t>(s->P) * g->nsl * g->nsl);
    int lb = 0;
    while ((int64_t(1) << lb) < want && lb < kAutoLogBuckets && lb < kb) ++lb;
    if (s->dw_log_buckets != 0) {
        if (s->dw_log_buckets < 1 || s->dw_log_buckets > kMaxLogBuckets || s->dw_log_buckets > kb) return SDM_ERR_SHAPE;
        lb = s->dw_log_buckets;
    }
    g->logB = lb;
    g->B = 1 << lb;
    // workspace: header | DW records [N, C*W] | bucket bounds [P, steps, B + 1]
    g->maxL = g->nk / kLongMin > 0 ? g->nk / kLongMin : 1;
    g->rstride = g->nk + g->maxL;
    if (N > (int64_t(1) << 31) / g->maxL) return SDM_ERR_SHAPE;   // long-group sum rows are int32-indexed
    g->krec_off = kHdrBytes;
    g->bb_off = g->krec_off + round_up(static_cast<size_t>(N) * g->rstride * sizeof(int4), 256);
    g->lcnt_off = g->bb_off + round_up(static_cast<size_t>(s->P) * (g->B + 1) * s->steps * sizeof(int32_t), 256);
    g->ldesc_off = g->lcnt_off + round_up(static_cast<size_t>(N) * sizeof(int32_t), 256);
    g->lacc_off = g->ldesc_off + round_up(static_cast<size_t>(N) * g->maxL * sizeof(int32_t), 256);
    g->ws_bytes = g->lacc_off + round_up(static_cast<size_t>(N) * g->maxL * s->hd * sizeof(float), 256);
    // Phase-1 shared memory: keys | vals | sidx | (pong + hist) or log-cumsums | pos | kb | rex | cpe | scratch
    const size_t np = static_cast<size_t>(g->npad);
    size_t off = 0;
    g->sm_keys = off;
    off += np * 4;
    g->sm_vals = off;
    off += np * (s->val_dtype == SDM_BF16 ? 2 : 4);
    g->sm_sidx = off;
    off += np * 2;
    g->sm_regd = off;
    g->sm_pong = off;
    off += np * 4;
    g->sm_pos = off;
    off += np * 4;
    g->sm_kb = off;
    off += np * 2;
    g->sm_rex = off;
    off += round_up(static_cast<size_t>(g->nk) * 4, 16);
    g->sm_tot = off;
    off += round_up(static_cast<size_t>(g->nk) * 4, 16);
    g->sm_kslot = off;
    off += round_up(static_cast<size_t>(g->nk) * 4, 16);
    // the DW bucket counters, and at least kHotExtra bytes: the dense pair path's vectors run on into
    // this region, idle by then
    g->sm_bcnt = off;
    off += std::max<size_t>(round_up((2 * static_cast<size_t>(g->B) + 1) * 4, 16), kHotExtra);
    // The dense pair path keeps its groups' vectors (3 * C floats each, after kHotMax 16-byte
    // descriptors) in the rex .. scratch region, free by then: the rex / cpe / write-row arrays and
    // the bucket-counter region. How many groups it takes must not depend on the launch geometry (the
    // DW bucket count changes that region), or other geometries would round some A / QK cells
    // differently: it is derived from the part every geometry has (3 arrays + kHotExtra).
    g->sm_zero = off;
    {
        const size_t room = 3 * round_up(static_cast<size_t>(g->nk) * 4, 16) + kHotExtra - kHotMax * 16;
        g->hot_cap = static_cast<int>(std::min<size_t>(kHotMax, room / (12 * static_cast<size_t>(g->C))));
    }
    // the sort's words go back and forth between the log-cumsum and the position-pack regions (idle
    // until the scans); its two digit-counter arrays ([digit][thread] uint16 each: 8 bytes per
    // position) lie over the regions from the write-before counts to the scratch (idle until the
    // scans; the bucket counters are zeroed after the sort), or after the scratch where those are
    // too small
    const size_t cnt_bytes = np * 8;
    g->sm_scr = off;
    off += 64 * 16 + 64 * 4;
    g->sm_hist = g->sm_kb;
    if (g->sm_kb + cnt_bytes > g->sm_scr) {
        g->sm_hist = round_up(off, 16);
        off = g->sm_hist + cnt_bytes;
    }
    g->smem_bytes = round_up(off, 128);
    return SDM_OK;
}

sdm_status check_ws(const Geometry& g, const void* ws, size_t ws_bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < g.ws_bytes) return SDM_ERR_WORKSPACE;
    return SDM_OK;
}

sdm_status check_range(const Geometry& g, int64_t b, int64_t e) {
    if (b < 0 || e > g.steps || b > e) return SDM_ERR_ARG;
    return SDM_OK;
}

sdm_status run_phase1(const sdm_shape* s, const Geometry& g, const int32_t* k_idx, const int32_t* q_idx,
                      const void* k_val, const void* q_val, const float* gate, const sdm_p1_out* out,
                      int64_t b, int64_t e, void* ws, cudaStream_t stream, int ordinals = 0) {
    P1Args a;
    memset(&a, 0, sizeof(a));
    a.k_idx = k_idx;
    a.q_idx = q_idx;
    a.k_val = k_val;
    a.q_val = q_val;
    a.g = gate;
    if (out != nullptr) a.out = *out;
    unsigned char* const w = static_cast<unsigned char*>(ws);
    a.krec = reinterpret_cast<int4*>(w + g.krec_off);
    a.bb = reinterpret_cast<int32_t*>(w + g.bb_off);
    a.lcnt = reinterpret_cast<int32_t*>(w + g.lcnt_off);
    a.ldesc = reinterpret_cast<int32_t*>(w + g.ldesc_off);
    a.maxL = g.maxL;
    a.rstride = g.rstride;
    a.status = reinterpret_cast<uint32_t*>(w + kHdrStatus);
    a.C = g.C;
    a.W = g.W;
    a.R = g.R;
    a.wr = g.wr;
    a.n = g.n;
    a.nk = g.nk;
    a.nq = g.nq;
    a.npad = g.npad;
    a.nwarps = g.nwarps;
    a.key_bits = g.key_bits;
    a.passes = g.passes;
    a.digit_bits = g.digit_bits;
    a.bucket_bits = g.bucket_bits;
    a.S = g.S;
    a.c0 = b * g.P;
    a.first_partial = (g.steps - 1) * g.P;
    a.valid_last = s->valid_last;
    a.g_width = s->gate_per_entry ? g.W : 1;
    a.g_lane_stride = s->gate_per_entry ? 1 : 0;
    a.wr_magic = static_cast<uint32_t>(((uint64_t(1) << 32) + g.wr - 1) / g.wr);
    a.w_magic = static_cast<uint32_t>(((uint64_t(1) << 32) + g.W - 1) / g.W);
    a.r_magic = static_cast<uint32_t>(((uint64_t(1) << 32) + g.R - 1) / g.R);
    a.P = g.P;
    a.logB = g.logB;
    a.steps = g.steps;
    a.sm_keys = static_cast<uint32_t>(g.sm_keys);
    a.sm_vals = static_cast<uint32_t>(g.sm_vals);
    a.sm_sidx = static_cast<uint32_t>(g.sm_sidx);
    a.sm_pong = static_cast<uint32_t>(g.sm_pong);
    a.sm_hist = static_cast<uint32_t>(g.sm_hist);
    a.sm_lv = static_cast<uint32_t>(g.sm_regd);
    a.sm_pos = static_cast<uint32_t>(g.sm_pos);
    a.sm_kb = static_cast<uint32_t>(g.sm_kb);
    a.sm_rex = static_cast<uint32_t>(g.sm_rex);
    a.sm_tot = static_cast<uint32_t>(g.sm_tot);
    a.sm_kslot = static_cast<uint32_t>(g.sm_kslot);
    a.sm_bcnt = static_cast<uint32_t>(g.sm_bcnt);
    a.sm_zero = static_cast<uint32_t>(g.sm_zero);
    a.hot_cap = g.hot_cap;
    a.sm_scr = static_cast<uint32_t>(g.sm_scr);
    const cudaError_t err =
        launch_phase1(a, s->val_dtype == SDM_BF16, ordinals, (e - b) * g.P, g.threads, g.smem_bytes, stream);
    return err == cudaSuccess ? SDM_OK : SDM_ERR_CUDA;
}

sdm_status run_dw(const sdm_shape* s, const Geometry& g, const void* dv, void* bank, void* snap, int64_t b, int64_t e,
                  void* ws, cudaStream_t stream) {
    unsigned char* const w = static_cast<unsigned char*>(ws);
    DWArgs a;
    memset(&a, 0, sizeof(a));
    a.krec = reinterpret_cast<const int4*>(w + g.krec_off);
    a.bb = reinterpret_cast<const int32_t*>(w + g.bb_off);
    a.lacc = reinterpret_cast<const float*>(w + g.lacc_off);
    a.dv = dv;
    a.bank = bank;
    a.snap = snap;
    a.claim = reinterpret_cast<uint32_t*>(w + kHdrClaim);
    a.P = g.P;
    a.C = g.C;
    a.W = g.W;
    a.nk = g.nk;
    a.maxL = g.maxL;
    a.rstride = g.rstride;
    a.B = g.B;
    a.nsl = g.nsl;
    a.hd = g.hd;
    a.S = g.S;
    a.steps = g.steps;
    a.step_begin = b;
    a.step_end = e;
    a.items = static_cast<int64_t>(g.P) * g.B * g.nsl;
    LongArgs la;   // the long groups' sums first (the DW takes them at their reference records)
    memset(&la, 0, sizeof(la));
    la.krec = a.krec;
    la.lcnt = reinterpret_cast<const int32_t*>(w + g.lcnt_off);
    la.ldesc = reinterpret_cast<const int32_t*>(w + g.ldesc_off);
    la.dv = dv;
    la.lacc = reinterpret_cast<float*>(w + g.lacc_off);
    la.claim = a.claim;   // the work counter starts at zero for every DW launch (the status word is kept)
    la.C = g.C;
    la.maxL = g.maxL;
    la.rstride = g.rstride;
    la.hd = g.hd;
    la.nsl = g.nsl;
    la.c0 = b * g.P;
    la.nchunks = (e - b) * g.P;
    if (launch_long(la, s->dv_dtype == SDM_BF16, stream) != cudaSuccess) return SDM_ERR_CUDA;
    const cudaError_t err = launch_dw(a, s->dv_dtype == SDM_BF16, s->bank_dtype == SDM_BF16, stream);
    return err == cudaSuccess ? SDM_OK : SDM_ERR_CUDA;
}

sdm_status check_p1_args(const Geometry& g, const int32_t* k_idx, const int32_t* q_idx, const void* k_val,
                         const void* q_val, const float* gate, const sdm_p1_out* out) {
    if (k_idx == nullptr || q_idx == nullptr || k_val == nullptr || q_val == nullptr || gate == nullptr) return SDM_ERR_ARG;
    if (!aligned16(k_idx) || !aligned16(q_idx) || !aligned16(k_val) || !aligned16(q_val) || !aligned16(gate))
        return SDM_ERR_ALIGN;
    if (out != nullptr) {
        const void* ptrs[] = {out->log_k, out->rex, out->cpe, out->k_eff, out->is_last, out->is_only,
                              out->pos_k, out->log_q, out->q_w, out->pos_q, out->q_last, out->q_only,
                              out->A, out->QK, out->sorted_k, out->sorted_q, out->repeats, out->ngroups};
        for (const void* p : ptrs)
            if (p != nullptr && !aligned16(p)) return SDM_ERR_ALIGN;
    }
    (void)g;
    return SDM_OK;
}

sdm_status check_smem(const Geometry& g) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SDM_ERR_CUDA;
    size_t lim = 0;
    if (phase1_smem_limit(dev, &lim) != cudaSuccess) return SDM_ERR_CUDA;
    // the kernel's static shared arrays (flag words, counters: under kP1StaticSmem) come on top
    return g.smem_bytes + kP1StaticSmem <= lim ? SDM_OK : SDM_ERR_SMEM;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" size_t sdm_workspace_bytes(const sdm_shape* shape) {
    Geometry g;
    if (geometry(shape, &g) != SDM_OK) return 0;
    return g.ws_bytes;
}

extern "C" sdm_status sdm_workspace_init(void* ws, size_t ws_bytes, sdm_stream_t stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < kHdrBytes)
        return SDM_ERR_WORKSPACE;
    return cudaMemsetAsync(ws, 0, kHdrBytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SDM_OK
                                                                                                    : SDM_ERR_CUDA;
}

extern "C" sdm_status sdm_phase1(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                                 const void* k_val, const void* q_val, const float* g, const sdm_p1_out* out,
                                 int64_t step_begin, int64_t step_end, void* ws, size_t ws_bytes,
                                 sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if ((st = check_p1_args(geo, k_idx, q_idx, k_val, q_val, g, out)) != SDM_OK) return st;
    if ((st = check_ws(geo, ws, ws_bytes)) != SDM_OK) return st;
    if ((st = check_smem(geo)) != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    return run_phase1(shape, geo, k_idx, q_idx, k_val, q_val, g, out, step_begin, step_end, ws,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" sdm_status sdm_dw(const sdm_shape* shape, const void* dv, void* bank, int64_t step_begin, int64_t step_end,
                             void* ws, size_t ws_bytes, sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if (dv == nullptr || bank == nullptr) return SDM_ERR_ARG;
    if (!aligned16(dv) || !aligned16(bank)) return SDM_ERR_ALIGN;
    if ((st = check_ws(geo, ws, ws_bytes)) != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    return run_dw(shape, geo, dv, bank, nullptr, step_begin, step_end, ws, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" sdm_status sdm_forward_chunks(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                                         const void* k_val, const void* q_val, const float* g, const void* dv,
                                         void* bank, const sdm_p1_out* out, int64_t step_begin, int64_t step_end,
                                         void* ws, size_t ws_bytes, sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if ((st = check_p1_args(geo, k_idx, q_idx, k_val, q_val, g, out)) != SDM_OK) return st;
    if (dv == nullptr || bank == nullptr) return SDM_ERR_ARG;
    if (!aligned16(dv) || !aligned16(bank)) return SDM_ERR_ALIGN;
    if ((st = check_ws(geo, ws, ws_bytes)) != SDM_OK) return st;
    if ((st = check_smem(geo)) != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = run_phase1(shape, geo, k_idx, q_idx, k_val, q_val, g, out, step_begin, step_end, ws, cs)) != SDM_OK)
        return st;
    return run_dw(shape, geo, dv, bank, nullptr, step_begin, step_end, ws, cs);
}

// ---- the saving forward: DW also writes the dense compact snapshot ------------------------------
extern "C" sdm_status sdm_phase1_saving(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                                        const void* k_val, const void* q_val, const float* g, const sdm_p1_out* out,
                                        int64_t step_begin, int64_t step_end, void* ws, size_t ws_bytes,
                                        sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if ((st = check_p1_args(geo, k_idx, q_idx, k_val, q_val, g, out)) != SDM_OK) return st;
    if ((st = check_ws(geo, ws, ws_bytes)) != SDM_OK) return st;
    if ((st = check_smem(geo)) != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    return run_phase1(shape, geo, k_idx, q_idx, k_val, q_val, g, out, step_begin, step_end, ws,
                      reinterpret_cast<cudaStream_t>(stream), 1);
}

extern "C" sdm_status sdm_dw_saving(const sdm_shape* shape, const void* dv, void* bank, void* snap, int64_t step_begin,
                                    int64_t step_end, void* ws, size_t ws_bytes, sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if (dv == nullptr || bank == nullptr || snap == nullptr) return SDM_ERR_ARG;
    if (!aligned16(dv) || !aligned16(bank) || !aligned16(snap)) return SDM_ERR_ALIGN;
    if ((st = check_ws(geo, ws, ws_bytes)) != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    return run_dw(shape, geo, dv, bank, snap, step_begin, step_end, ws, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" sdm_status sdm_forward_chunks_saving(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                                                const void* k_val, const void* q_val, const float* g, const void* dv,
                                                void* bank, void* snap, const sdm_p1_out* out, int64_t step_begin,
                                                int64_t step_end, void* ws, size_t ws_bytes, sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if ((st = check_p1_args(geo, k_idx, q_idx, k_val, q_val, g, out)) != SDM_OK) return st;
    if (dv == nullptr || bank == nullptr || snap == nullptr) return SDM_ERR_ARG;
    if (!aligned16(dv) || !aligned16(bank) || !aligned16(snap)) return SDM_ERR_ALIGN;
    if ((st = check_ws(geo, ws, ws_bytes)) != SDM_OK) return st;
    if ((st = check_smem(geo)) != SDM_OK) return st;
    if (step_begin == step_end) return SDM_OK;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = run_phase1(shape, geo, k_idx, q_idx, k_val, q_val, g, out, step_begin, step_end, ws, cs, 1)) != SDM_OK)
        return st;
    return run_dw(shape, geo, dv, bank, snap, step_begin, step_end, ws, cs);
}

// ---- the no-allocation forward ----------------------------------------------------------------
// Scratch for callers that cannot allocate device memory: a file-scope device array that every GPU
// loading this library holds until the process exits. Host code must not use the array's name as a
// device address: its address is looked up with cudaGetSymbolAddress, on every call made outside a
// stream capture (a device context created again after cudaDeviceReset gets a new address) and
// remembered per device for calls made inside a capture.
namespace {
__device__ __align__(256) unsigned char g_noalloc_scratch[SDM_NOALLOC_SCRATCH_BYTES];
constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

sdm_status noalloc_scratch(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SDM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SDM_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SDM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (cap == cudaStreamCaptureStatusNone || g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SDM_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SDM_OK;
}
}  // namespace

extern "C" sdm_status sdm_forward_chunks_noalloc(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                                                 const void* k_val, const void* q_val, const float* g, const void* dv,
                                                 void* bank, const sdm_p1_out* out, int64_t step_begin,
                                                 int64_t step_end, int32_t* status_out, sdm_stream_t stream) {
    Geometry geo;
    sdm_status st = geometry(shape, &geo);
    if (st != SDM_OK) return st;
    if ((st = check_range(geo, step_begin, step_end)) != SDM_OK) return st;
    if ((st = check_p1_args(geo, k_idx, q_idx, k_val, q_val, g, out)) != SDM_OK) return st;
    if (dv == nullptr || bank == nullptr) return SDM_ERR_ARG;
    if (!aligned16(dv) || !aligned16(bank)) return SDM_ERR_ALIGN;
    if (geo.ws_bytes > SDM_NOALLOC_SCRATCH_BYTES) return SDM_ERR_WORKSPACE;
    if ((st = check_smem(geo)) != SDM_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    if ((st = noalloc_scratch(cs, &ws)) != SDM_OK) return st;
    // the scratch keeps the previous call's bytes: the status word and the work counter restart at 0
    if (cudaMemsetAsync(ws, 0, kHdrBytes, cs) != cudaSuccess) return SDM_ERR_CUDA;
    if (step_begin < step_end) {
        if ((st = run_phase1(shape, geo, k_idx, q_idx, k_val, q_val, g, out, step_begin, step_end, ws, cs)) != SDM_OK)
            return st;
        if ((st = run_dw(shape, geo, dv, bank, nullptr, step_begin, step_end, ws, cs)) != SDM_OK) return st;
    }
    if (status_out != nullptr &&
        cudaMemcpyAsync(status_out, static_cast<unsigned char*>(ws) + kHdrStatus, sizeof(int32_t),
                        cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
        return SDM_ERR_CUDA;
    return SDM_OK;
}

extern "C" sdm_status sdm_device_status(const void* ws, int32_t* code_out, int32_t clear, sdm_stream_t stream) {
    if (ws == nullptr || code_out == nullptr) return SDM_ERR_ARG;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, static_cast<const unsigned char*>(ws) + kHdrStatus, sizeof(word), cudaMemcpyDeviceToHost,
                        cs) != cudaSuccess)
        return SDM_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return SDM_ERR_CUDA;
    *code_out = static_cast<int32_t>(word);
    if (clear && word != 0u) {
        if (cudaMemsetAsync(const_cast<void*>(ws), 0, sizeof(word), cs) != cudaSuccess) return SDM_ERR_CUDA;
        if (cudaStreamSynchronize(cs) != cudaSuccess) return SDM_ERR_CUDA;
    }
    return word == 0u ? SDM_OK : SDM_ERR_DEVICE;
}

extern "C" const char* sdm_status_string(sdm_status status) {
    switch (status) {
        case SDM_OK: return "SDM_OK";
        case SDM_ERR_ARG: return "SDM_ERR_ARG: a required pointer is NULL or a step range is invalid";
        case SDM_ERR_SHAPE: return "SDM_ERR_SHAPE: a size is outside the supported limits";
        case SDM_ERR_DTYPE: return "SDM_ERR_DTYPE: unknown dtype code";
        case SDM_ERR_ALIGN: return "SDM_ERR_ALIGN: a pointer is not 16-byte aligned or hd % 4 != 0";
        case SDM_ERR_WORKSPACE: return "SDM_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case SDM_ERR_SMEM: return "SDM_ERR_SMEM: the chunk does not fit the device's shared memory";
        case SDM_ERR_CUDA: return "SDM_ERR_CUDA: a CUDA runtime call failed";
        case SDM_ERR_DEVICE: return "SDM_ERR_DEVICE: the device status word is nonzero";
    }
    return "unknown sdm_status";
}
