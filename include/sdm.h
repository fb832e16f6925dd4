/*
 * sdm.h -- C ABI of the GB300 (sm_103a) hot path of the chunked sparse-delta-memory (SDM)
 * recurrence: the forward's Phase 1 and Phase-2 decay-and-write (DW), the saving forward's dense
 * snapshot, and the deterministic backward's step kernels (Phase A, GWR, GDS).
 *
 * Definitions followed (sparse-delta-memory 2.0.0):
 *   phase1_cuda.py, module docstring ........ the Phase-1 outputs and the determinism contract
 *   phase1_cuda.py, p1_keys_zw_kernel ........ entry order and payload bits, invalid tokens
 *   phase1_cuda.py, p1_scan_kernel ........... gates, log-cumsums, rex, cpe, flags, pos pack,
 *                                              sorted-row elements
 *   phase1_cuda.py, p1_pairs_kernel comment .. the A / QK pair triangles
 *   mover_da2_cuda.py, module docstring ...... DW: bank[s] = fma(base, cpe_last, acc),
 *                                              acc = fma(sc_m, dv[tok_m], acc) in sorted order
 *   mover_fx_cuda.py, module docstring ....... the bank-direct DW contract (base read from the
 *                                              bank row itself; one writer per row and launch)
 *   pa_dc_cuda.py, module docstring .......... the backward step: Phase A (the backward of DW)
 *                                              and GWR (the write side's token gather)
 *   mover_da2_cuda.py, "GDS, split by data need" the backward's read side (dots and scatter)
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer owned by the caller. The library never allocates
 *     device or host memory. It launches on `stream` and never synchronizes it (except
 *     sdm_device_status, which reads a word back).
 *   - Layout is chunk-major: chunk c = ti * P + p holds tokens [ti*C, (ti+1)*C) of stream p,
 *     for ti in [0, steps). N = steps * P chunks.
 *       k_idx [N, C, W] int32, q_idx [N, C, R] int32: stream-local slot ids in [0, S). Ids of
 *         invalid tokens (t >= valid_last in the last step's chunks) are ignored.
 *       k_val [N, C, W], q_val [N, C, R]: val_dtype (float32 or bfloat16).
 *       g: float32 [N, C] one gate per token (gate_per_entry = 0) or [N, C, W] per write entry (1).
 *       dv [N * C, hd]: dv_dtype; row c * C + t is token t of chunk c.
 *       bank [P * S, hd]: bank_dtype; stream p owns rows [p*S, (p+1)*S). Updated in place.
 *   - Alignment: bank, dv and every output array 16-byte aligned; hd a multiple of 4.
 *   - Limits: 1 <= C <= 256, 1 <= W, R <= 256, C * (W + R) <= 8192 (one chunk sorts on chip),
 *     1 <= S <= 2^31 - 1, P * S * hd fits in int64.
 *   - Shape, dtype, alignment and workspace errors are returned BEFORE any launch. Errors the
 *     device finds (a valid slot id outside [0, S)) are OR-ed into a status word inside the
 *     workspace (read it with sdm_device_status), or, for the backward entry points, into the
 *     caller's optional status word. No kernel traps, and no kernel waits on another thread block.
 *   - Determinism: for fixed inputs, shapes and GPU type every output is bitwise reproducible.
 *     The sort is stable, scans combine in a fixed tree, every A/QK cell and every bank row has
 *     one writer that adds its terms in an input-determined order, and no atomics touch a sum.
 */
#ifndef SDM_H
#define SDM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* sdm_stream_t;

typedef enum {
    SDM_OK = 0,
    SDM_ERR_ARG = -1,       /* a required pointer is NULL, or a step range is reversed / out of range */
    SDM_ERR_SHAPE = -2,     /* a size is outside the limits above */
    SDM_ERR_DTYPE = -3,     /* an unknown dtype code */
    SDM_ERR_ALIGN = -4,     /* a pointer is not 16-byte aligned, or hd % 4 != 0 */
    SDM_ERR_WORKSPACE = -5, /* ws is NULL, misaligned or smaller than sdm_workspace_bytes */
    SDM_ERR_SMEM = -6,      /* the chunk does not fit the device's shared memory */
    SDM_ERR_CUDA = -7,      /* a CUDA runtime call failed (launch, attribute, memset) */
    SDM_ERR_DEVICE = -8     /* sdm_device_status found a nonzero device status word */
} sdm_status;

typedef enum { SDM_F32 = 0, SDM_BF16 = 1 } sdm_dtype;

/* Bits of the device status word (sdm_device_status). */
#define SDM_DEV_BAD_SLOT 0x1u /* a valid entry's slot id was outside [0, S): the entry is dropped */

typedef struct {
    int32_t P;              /* streams */
    int32_t C;              /* tokens per chunk */
    int32_t W;              /* write (K) entries per token */
    int32_t R;              /* read (Q) entries per token */
    int32_t hd;             /* bank / dv row width */
    int32_t valid_last;     /* valid tokens of the last step's chunks, 1..C */
    int64_t steps;          /* chunks per stream */
    int64_t S;              /* slots per stream */
    int32_t val_dtype;      /* sdm_dtype of k_val, q_val and of cpe / k_eff / q_w */
    int32_t dv_dtype;       /* sdm_dtype of dv */
    int32_t bank_dtype;     /* sdm_dtype of the bank */
    int32_t gate_per_entry; /* 0: g [N, C]; 1: g [N, C, W] */
    /* Launch geometry of the forward's kernels, 0 = chosen from the shape (the backward's entry
     * points ignore both). Neither changes any output bit (every sum is taken in an order fixed by
     * the input), only how the work is split:
     *   dw_log_buckets 1..11 (<= ceil(log2 S)): the DW walk's hashed slot buckets per stream, 2^k
     *                  (changes sdm_workspace_bytes and Phase 1's shared memory per block: 8 bytes a
     *                  bucket); 0 = about 32768 / ceil(hd / 128) DW work items per launch, at most 2^10
     *                  buckets;
     *   p1_warps       the automatic count .. 32: warps of a Phase-1 block (extra warps hold
     *                  padding entries; more shared memory per block). */
    int32_t dw_log_buckets;
    int32_t p1_warps;
} sdm_shape;

/*
 * Phase-1 outputs, entry order (phase1_cuda.py module docstring and p1_scan_kernel). Any field
 * may be NULL: it is not written.
 *   [N, C, W]: log_k f32 (log-cumsum of the slot's gates at the entry, own token included),
 *              rex f32 (gates of the slot's later writes in the chunk), cpe val_dtype
 *              (exp of the slot's total gate in the chunk), k_eff val_dtype (k * exp(log_k)),
 *              is_last / is_only int8, pos_k int32 (position pack below).
 *   [N, C, R]: log_q f32, q_w val_dtype (q * exp(log_q)), pos_q int32, q_last / q_only int8.
 *   A, QK [N, C, C] f32: A[i][j] = sum over shared slots of k_i k_j exp(log_k_i - log_k_j),
 *              j < i; QK[i][j] = sum of q_i k_j exp(log_q_i - log_k_j), j <= i; zero elsewhere.
 *   sorted_k [N, C*W], sorted_q [N, C*R] int32: each kind's entries in sorted order as
 *              (entry bits: lane | isQ << 8 | token << 9 | invalid << 17)
 *              | min(peers before, 4095) << 18 | LAST << 30 | FIRST << 31; invalid: | 3 << 30.
 *   repeats: one int64 to which the count of repeated write entries (a token's write entry on
 *            a slot its previous write entry of the group already holds) is ADDED.
 *   ngroups [N] int32: the chunk's valid write groups (slots with at least one valid write
 *            entry), i.e. the rows of its dense compact snapshot; written only by the saving
 *            forward's Phase 1 (sdm_phase1_saving, sdm_forward_chunks_saving).
 *   stats [4] int64: counters of the call's chunks, ADDED to (the caller zeroes them): [0] valid
 *            write groups (slot groups with at least one valid write entry: the DW's base-row reads
 *            and row writes), [1] slot groups whose pair terms took the dense rank-1 path, [2] pair
 *            terms summed one by one (an entry and an earlier write entry of its group, into A or
 *            QK), [3] A / QK rows the pair phase writes (a token's row in a triangle where one of its
 *            entries has an earlier valid write entry in its group, or that a dense group
 *            reaches). [1..3] are counted only when A or QK is requested. Diagnostic counters in the manner of phase1_cuda.py's repeats counter.
 * Position pack: r | min(after, 127) << 17 | min(before + 1 + min(after, 127), 127) << 24 for a
 * valid entry (r = position in the chunk's sorted row, before / after = valid entries of the
 * same kind and slot before / after it), r alone for an invalid entry. Invalid entries:
 * log 0, rex 0, cpe 1, k_eff / q_w 0, flags 0.
 */
typedef struct {
    float* log_k;
    float* rex;
    void* cpe;
    void* k_eff;
    int8_t* is_last;
    int8_t* is_only;
    int32_t* pos_k;
    float* log_q;
    void* q_w;
    int32_t* pos_q;
    int8_t* q_last;
    int8_t* q_only;
    float* A;
    float* QK;
    int32_t* sorted_k;
    int32_t* sorted_q;
    int64_t* repeats;
    int32_t* ngroups;
    int64_t* stats;
} sdm_p1_out;

/*
 * Bytes of the caller-allocated device workspace for this shape: a 256-byte header (status word,
 * DW work counter), the DW records of every chunk (16 bytes per write entry) and the per-chunk
 * slot-bucket bounds of the DW work split. The workspace must be 256-byte aligned and, before its
 * first use, initialised with sdm_workspace_init. One workspace serves one stream of calls at a
 * time. Returns 0 for an invalid shape.
 */
size_t sdm_workspace_bytes(const sdm_shape* shape);

/* Zeroes the workspace's header (status word and work counter) on `stream`. */
sdm_status sdm_workspace_init(void* ws, size_t ws_bytes, sdm_stream_t stream);

/*
 * Phase 1 of the chunks of steps [step_begin, step_end) (all P streams): the outputs in `out`
 * and, in `ws`, the DW records of those chunks. Inputs are the full [N, ...] arrays; only the
 * range's chunks are read and written. Launches one kernel (one CTA per chunk).
 */
sdm_status sdm_phase1(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                      const void* k_val, const void* q_val, const float* g, const sdm_p1_out* out,
                      int64_t step_begin, int64_t step_end, void* ws, size_t ws_bytes,
                      sdm_stream_t stream);

/*
 * DW of steps [step_begin, step_end), in step order, from the records sdm_phase1 left in `ws`
 * for those steps: per slot group of each chunk, bank[p*S + s] = fma(base, cpe_last, acc),
 * acc = fma(sc_m, dv[tok_m], acc) over the group's write entries in sorted order starting at 0,
 * sc = f32(k) * expf(rex), base = the row before this step (stored RN in bfloat16, or as the f32
 * result). One launch runs every step: each warp owns a range of slots of one stream and applies
 * the range's groups of all steps in order, so no warp ever waits for another.
 */
sdm_status sdm_dw(const sdm_shape* shape, const void* dv, void* bank, int64_t step_begin,
                  int64_t step_end, void* ws, size_t ws_bytes, sdm_stream_t stream);

/*
 * The forward over steps [step_begin, step_end): sdm_phase1 then sdm_dw on `stream`.
 * `out` may be NULL (no Phase-1 outputs written; records still go to ws). Running [0, k) then
 * [k, steps) gives the same bits as [0, steps).
 */
sdm_status sdm_forward_chunks(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                              const void* k_val, const void* q_val, const float* g, const void* dv,
                              void* bank, const sdm_p1_out* out, int64_t step_begin,
                              int64_t step_end, void* ws, size_t ws_bytes, sdm_stream_t stream);

/*
 * Phase 1 of the saving forward: sdm_phase1, and in addition each group's FIRST DW record carries
 * the group's dense ordinal (below) and out->ngroups is written. Its records serve sdm_dw_saving
 * (and sdm_dw); the records of sdm_phase1 serve sdm_dw only. Errors: those of sdm_phase1.
 */
sdm_status sdm_phase1_saving(const sdm_shape* shape, const int32_t* k_idx, const int32_t* q_idx,
                             const void* k_val, const void* q_val, const float* g,
                             const sdm_p1_out* out, int64_t step_begin, int64_t step_end, void* ws,
                             size_t ws_bytes, sdm_stream_t stream);

/*
 * The saving forward's DW (mover_fx_cuda.py, module docstring; mover_da2_cuda.py, the WR mode of the
 * DW walk): sdm_dw, and in addition every valid write group's base row -- the bank row before this
 * step's write, as raw bytes of the bank type -- goes to the dense compact snapshot
 *   snap [N, C*W, hd] (bank dtype, 16-byte aligned, caller-owned), row c * (C*W) + g,
 * g = the group's dense ordinal in chunk c: the number of the chunk's valid write groups (slots with
 * at least one valid write entry) before it in sorted order, i.e. slots ascending. Rows g >=
 * ngroups[c] (sdm_p1_out.ngroups) are not written. The records must come from sdm_phase1_saving
 * (they carry the ordinals). Bank results are those of sdm_dw, bit for bit.
 * Errors: those of sdm_dw; snap NULL -> SDM_ERR_ARG, misaligned -> SDM_ERR_ALIGN.
 */
sdm_status sdm_dw_saving(const sdm_shape* shape, const void* dv, void* bank, void* snap,
                         int64_t step_begin, int64_t step_end, void* ws, size_t ws_bytes,
                         sdm_stream_t stream);

/* sdm_phase1_saving then sdm_dw_saving on `stream` (arguments as sdm_forward_chunks, plus snap). */
sdm_status sdm_forward_chunks_saving(const sdm_shape* shape, const int32_t* k_idx,
                                     const int32_t* q_idx, const void* k_val, const void* q_val,
                                     const float* g, const void* dv, void* bank, void* snap,
                                     const sdm_p1_out* out, int64_t step_begin, int64_t step_end,
                                     void* ws, size_t ws_bytes, sdm_stream_t stream);

/* Bytes of the library-owned scratch used by sdm_forward_chunks_noalloc (16 MiB). */
#define SDM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * The forward of sdm_forward_chunks for callers that cannot allocate device memory -- for example
 * code inside a host framework that owns every device allocation, or a plugin interface that is
 * handed only its input and output buffers. It takes no workspace: it uses a scratch array of
 * SDM_NOALLOC_SCRATCH_BYTES compiled into the library (every GPU that loads the library holds it
 * until the process exits). It calls no cudaMalloc / cudaFree and no allocating library routine.
 * The pages (sparse-delta-memory 2.0.0) have no counterpart of this entry point.
 *   - Arguments and results are those of sdm_forward_chunks, without ws / ws_bytes.
 *   - Shapes whose workspace (sdm_workspace_bytes) exceeds SDM_NOALLOC_SCRATCH_BYTES are rejected
 *     with SDM_ERR_WORKSPACE before any launch; use sdm_forward_chunks with a caller workspace.
 *   - status_out (nullable): one device int32 that receives the call's device status word
 *     (SDM_DEV_* bits, 0 = fine), copied on `stream` after the kernels.
 *   - A call outside stream capture looks up the scratch's device address (with the calling
 *     thread's current device), so a device context created again (after cudaDeviceReset) is
 *     picked up; a call inside a stream capture reuses the address of the last call on that device
 *     outside capture: make at least one call before any capture, and again after a device reset.
 *   - Every call shares the one scratch and clears its header first. Calls whose kernels overlap
 *     on the GPU (different streams, or concurrent host threads) race on it: serialize them.
 */
sdm_status sdm_forward_chunks_noalloc(const sdm_shape* shape, const int32_t* k_idx,
                                      const int32_t* q_idx, const void* k_val, const void* q_val,
                                      const float* g, const void* dv, void* bank,
                                      const sdm_p1_out* out, int64_t step_begin, int64_t step_end,
                                      int32_t* status_out, sdm_stream_t stream);

/*
 * The forward's read-side token gather (mover_fx_cuda.py: fx_fwd_steps, each step's gather before its
 * dual matmul and DW; the weighted read whose vector-Jacobian product in q_w is the GDS dot
 * d_q_w[t, r] = <gr[t], bank[slot]> of mover_da2_cuda.py's module docstring; the token_gather form of
 * GWR's d_delta_v, pa_dc_cuda.py's module docstring), for every chunk c = ti * P + p of steps
 * [step_begin, step_end):
 *   y[c, t] = acc, acc = 0; acc = fmaf(q_w[c, t, r], bank[p*S + q_idx[c, t, r]], acc) over the read
 *   lanes r = 0 .. R-1 in order (float32; a lane whose id lies outside [0, S) adds nothing) for valid
 *   tokens t; padding tokens (t >= valid_last in the last step) get zeros.
 *   q_idx [N, C, R] int32, q_w [N, C, R] val_dtype (Phase 1's q_w output, or any weights),
 *   bank [P*S, hd] bank_dtype, read only: the rows as they are when the kernel runs, so a range of
 *   several steps reads one bank state (the forward's order is the caller's: the read of step t, then
 *   the DW of step t); y [N, C, hd] float32, only the range's chunks written. The pages' "dual matmul"
 *   (the chunk-internal part of the read, from A / QK) is not printed there and is not provided.
 *   status (nullable): SDM_DEV_BAD_SLOT is OR-ed when a valid token reads an id outside [0, S).
 * Errors: the shape's (SDM_ERR_SHAPE / DTYPE / ALIGN for hd % 4), SDM_ERR_ARG (step range, null
 * q_idx / q_w / bank / y), SDM_ERR_ALIGN (bank or y not 16-byte aligned), before any launch.
 * One launch (resident warps looping over (token, 128-column slice) units).
 */
sdm_status sdm_read(const sdm_shape* shape, const int32_t* q_idx, const void* q_w, const void* bank, float* y,
                    int64_t step_begin, int64_t step_end, uint32_t* status, sdm_stream_t stream);

/*
 * Phase A of the backward (pa_dc_cuda.py, module docstring: "PA per write group"; records kernel):
 * the backward of DW for the steps [step_begin, step_end), LAST step first (one launch per step;
 * step ti reads the grad rows step ti + 1 wrote). Per valid write group of chunk c = ti * P + p
 * (slot s, members m in sorted order, as sorted_k lists them):
 *   sc_m = -beta[c, tok_m] * (f32(k_m) * expf(log_k_m))
 *   acc = 0; acc = fmaf(sc_m, dva[c, tok_m], acc) over the members in order
 *   grad[p*S + s] = RN(fmaf(gdw, cpe_last, acc))    gdw = the row before this step, cpe_last = cpe of
 *                                                    the group's last member (f32 grad: the fmaf itself)
 *   bank[p*S + s] = the group's snapshot row        (raw bytes: the row before the forward's write)
 *   grad_g[e] = cpe_e * <gdw, snap>,  d_k_eff[e] = -beta[c, tok_e] * <dva[c, tok_e], snap>
 * Dots are f32: per lane an fmaf chain over 4 columns of a 128-column slice, an xor butterfly over
 * the 32 lanes, slices added in order, so results do not depend on the launch geometry.
 * Arguments (device pointers, 16-byte aligned, caller-owned; shapes use `shape`'s N = steps * P):
 *   grad_dtype: sdm_dtype of grad (SDM_F32, or SDM_BF16 for grad rows in the bank's format).
 *   sorted_k [N, C*W] int32: as sdm_phase1 writes it (entries whose slot is outside [0, S) are
 *            invalid there). log_k f32 / cpe val_dtype [N, C, W]: sdm_phase1's outputs.
 *   k_idx int32 / k_val val_dtype [N, C, W]: the forward's inputs. beta f32 [N, C].
 *   dva f32 [N, C, hd]: the gradient of the forward's token rows (dv) for these steps.
 *   grad [P*S, hd] grad_dtype, bank [P*S, hd] bank_dtype: updated in place.
 *   snap: the dense compact snapshot rows of the steps in range, [step_end - step_begin, P, C*W, hd]
 *         in the bank dtype: row ((ti - step_begin) * P + p) * C*W + g for the group of dense ordinal g
 *         (sdm_dw_saving's layout; a caller holding all N chunks passes its row step_begin * P * C*W).
 *   d_k_eff, grad_g [N, C, W] f32: written for every entry of the range's chunks (0 for invalid
 *         entries).
 *   status (nullable): device word OR-ed with SDM_DEV_BAD_SLOT when a group's slot (k_idx of its
 *         first member) lies outside [0, S); the group is then skipped.
 * Errors: SDM_ERR_SHAPE / SDM_ERR_DTYPE / SDM_ERR_ALIGN for the shape (as sdm_phase1), grad_dtype
 * not 0 or 1 -> SDM_ERR_DTYPE, a NULL array -> SDM_ERR_ARG, a misaligned array -> SDM_ERR_ALIGN, a
 * bad step range -> SDM_ERR_ARG, a failed launch -> SDM_ERR_CUDA. No launch happens on an error
 * found before the first launch.
 */
sdm_status sdm_pa(const sdm_shape* shape, int32_t grad_dtype, const int32_t* sorted_k, const int32_t* k_idx,
                  const void* k_val, const float* log_k, const void* cpe, const float* beta, const float* dva,
                  void* grad, void* bank, const void* snap, float* d_k_eff, float* grad_g, int64_t step_begin,
                  int64_t step_end, uint32_t* status, sdm_stream_t stream);

/*
 * GWR, the token gather of the write side of the backward (pa_dc_cuda.py: module docstring, "GWR",
 * and its GWR kernel), for the steps [step_begin, step_end), LAST step first (one launch per step).
 * Per chunk c = ti * P + p and valid token t (t < valid_last in the last step's chunks, else t < C):
 *   d_delta_v[c, t] = acc, acc = 0; acc = fmaf(write_w[c, t, n], grad[p*S + k_idx[c, t, n]], acc)
 *                     over the write lanes n = 0 .. W-1 in order;
 *   d_k_pd[c, t, n] = <dv[c*C + t], grad[p*S + k_idx[c, t, n]]>  (f32 dots as sdm_pa's);
 * padding tokens get zero rows and zero dots.
 * Arguments (device pointers, 16-byte aligned, caller-owned; N = steps * P):
 *   grad_dtype: sdm_dtype of grad. k_idx int32 [N, C, W]: the forward's write ids. write_w f32
 *   [N, C, W]: the write weights. dv [N*C, hd] dv_dtype: the forward's token rows. grad [P*S, hd]
 *   grad_dtype: read only. d_delta_v f32 [N, C, hd], d_k_pd f32 [N, C, W]: written for the range.
 *   status (nullable): device word OR-ed with SDM_DEV_BAD_SLOT when a valid token's write id lies
 *   outside [0, S) (that lane adds nothing and its dot is 0).
 * Errors: as sdm_pa.
 */
sdm_status sdm_gwr(const sdm_shape* shape, int32_t grad_dtype, const int32_t* k_idx, const float* write_w,
                   const void* dv, const void* grad, float* d_delta_v, float* d_k_pd, int64_t step_begin,
                   int64_t step_end, uint32_t* status, sdm_stream_t stream);

/*
 * GDS, the read side of the backward (mover_da2_cuda.py: module docstring, the "GDS, split by data
 * need" comment, its read-records kernel), for the steps [step_begin, step_end), LAST step first
 * (two launches per step: the dots, then the scatter). Per chunk c = ti * P + p:
 *   d_q_w[c, t, r] = <gr[c, t], bank[p*S + q_idx[c, t, r]]> for the valid tokens t (t < valid_last
 *                   in the last step's chunks, else t < C); 0 for padding tokens;
 *   per read group (slot s with valid read entries; members m in sorted order as sorted_q lists them)
 *   acc = 0; acc = fmaf(sc_m, gr[c, tok_m], acc), sc = f32(q_m) * expf(log_q_m);
 *   grad[p*S + s] = RN(grad[p*S + s] + acc)          (one rounding per element; f32 grad: the sum)
 * Dots are f32 like sdm_pa's (per-lane fmaf chain over 4 columns, a fixed lane tree, slices in
 * order), so results do not depend on the launch geometry; every grad row has one writer per launch.
 * Arguments (device pointers, 16-byte aligned, caller-owned; N = steps * P):
 *   grad_dtype: sdm_dtype of grad (SDM_F32, or SDM_BF16 for grad rows in the bank's format).
 *   sorted_q [N, C*R] int32: as sdm_phase1 writes it. log_q f32 [N, C, R]: sdm_phase1's output.
 *   q_idx int32 / q_val val_dtype [N, C, R]: the forward's inputs. gr f32 [N, C, hd]: the gradient of
 *   the read results. bank [P*S, hd] bank_dtype: read only. grad [P*S, hd] grad_dtype: updated in
 *   place (must not alias bank). d_q_w [N, C, R] f32: written for every read entry of the range.
 *   status (nullable): device word OR-ed with SDM_DEV_BAD_SLOT when a valid token's read id lies
 *   outside [0, S) (its dot is 0 and it adds nothing).
 * Errors: as sdm_pa.
 */
sdm_status sdm_gds(const sdm_shape* shape, int32_t grad_dtype, const int32_t* sorted_q, const int32_t* q_idx,
                   const void* q_val, const float* log_q, const float* gr, const void* bank, void* grad, float* d_q_w,
                   int64_t step_begin, int64_t step_end, uint32_t* status, sdm_stream_t stream);

/*
 * Synchronizes `stream`, reads the workspace's device status word into *code_out (0 = fine,
 * else SDM_DEV_* bits) and, if `clear`, zeroes it. Returns SDM_ERR_DEVICE when the word is
 * nonzero, SDM_ERR_CUDA when the copy fails.
 */
sdm_status sdm_device_status(const void* ws, int32_t* code_out, int32_t clear, sdm_stream_t stream);

/* A static string naming a status code. */
const char* sdm_status_string(sdm_status status);

#ifdef __cplusplus
}
#endif

#endif /* SDM_H */
