/*
 * sdm_oracle.c -- plain, slow, float64 CPU oracle of the sparse-delta-memory forward hot path:
 * Phase 1 (stable sort by slot, segmented log-cumsums, flags, packed positions, sorted rows,
 * pair triangles) and the Phase-2 decay-and-write (DW).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call this file; only
 * the tests, the package's smoke check and the benchmark's CPU-baseline leg use it. It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * Sources (sparse-delta-memory 2.0.0):
 *  - phase1_cuda.py, module docstring: the Phase-1 outputs (log_k, log_q, rex, cpe, is_last,
 *    is_only, k_eff, q_w, A, QK, pos_k, pos_q, q_last, q_only) and the determinism contract.
 *  - phase1_cuda.py, p1_keys_zw_kernel: entry order (per token W write columns, then R read
 *    columns), the payload bits and invalid tokens (t >= valid_last in the partial chunks).
 *  - phase1_cuda.py, p1_scan_kernel: the gate x of an entry (write entries only, a token's
 *    repeated write entry of one slot contributes 0), inclusive log-cumsum, rex = gates after,
 *    cpe = exp(group total) in the value type, the position pack and the sorted-row element.
 *  - phase1_cuda.py, p1_pairs_kernel comment: which (entry, earlier write entry) pairs add a
 *    term to A (write x write, other token) and to QK (read x write, same token allowed).
 *  - mover_da2_cuda.py and mover_fx_cuda.py module docstrings: the DW per-group update
 *    bank[s] = base * cpe_last + sum_m k_m * exp(rex_m) * dv[tok_m], cpe as stored in the value type.
 *
 * Everything is computed in float64; values the method stores in a narrower type are returned
 * unrounded (the caller compares them within that type's tolerance), except where the pages
 * make a rounded value an input of a later step (cpe feeds DW as stored; the bank row is
 * stored in the bank type between steps), which the DW routine reproduces on request.
 *
 * Pins (tests/test_oracle_pins.py): brute-force pair sums over lane pairs, a token-sequential
 * bank recurrence, brute-force sort positions, closed forms for rex/cpe and flag invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- rounding to the storage types ------------------------------------------------------ */

/* Round to the nearest bfloat16 value (8 significant bits, ties to even). */
static double round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    double m = frexp(x, &e); /* x = m * 2^e, 0.5 <= |m| < 1 */
    int shift = 8;
    if (e - 8 < -133) shift = e + 133; /* bfloat16 subnormal spacing 2^-133 */
    double r = nearbyint(ldexp(m, shift));
    return ldexp(r, e - shift);
}

static double round_f32(double x) { return (double)(float)x; }

static double round_to(double x, int bf16) { return bf16 ? round_bf16(x) : round_f32(x); }

/* ---- one chunk: entries, stable sort by slot, groups --------------------------------------- */

typedef struct {
    int64_t key;
    int32_t e;
} ent_t;

static int cmp_ent(const void* a, const void* b) {
    const ent_t* x = (const ent_t*)a;
    const ent_t* y = (const ent_t*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return x->e < y->e ? -1 : (x->e > y->e); /* index order breaks ties: a stable sort */
}

typedef struct {
    int C, W, R, V, n;
    /* by entry e = t * (W + R) + j */
    int *tok, *lane, *isq, *valid, *rank, *gstart, *gend;
    int64_t* slot;
    double *val, *x, *logv, *rex, *gtot, *gabs;
    int *kb, *ka, *qb, *qa, *rep;
    /* by sorted position r */
    int* order;
    ent_t* ents;
} chunk_t;

static void chunk_free(chunk_t* ch) {
    free(ch->tok); free(ch->lane); free(ch->isq); free(ch->valid); free(ch->rank);
    free(ch->gstart); free(ch->gend); free(ch->slot); free(ch->val); free(ch->x); free(ch->logv);
    free(ch->rex); free(ch->gtot); free(ch->gabs); free(ch->kb); free(ch->ka); free(ch->qb);
    free(ch->qa); free(ch->rep); free(ch->order); free(ch->ents);
}

/* Builds the entry list of one chunk and everything Phase 1 derives per entry.
 * g_width / g_lane_stride: the gate of (token t, write lane a) is g[t * g_width + a * g_lane_stride].
 * Returns 0, or -1 when a valid entry's slot is outside [0, S). */
static int chunk_analyze(chunk_t* ch, int C, int W, int R, int V, int64_t S, const int32_t* k_idx,
                         const int32_t* q_idx, const double* k_val, const double* q_val,
                         const double* g, int g_width, int g_lane_stride) {
    const int wr = W + R, n = C * wr;
    memset(ch, 0, sizeof(*ch));
    ch->C = C; ch->W = W; ch->R = R; ch->V = V; ch->n = n;
#define ALLOC(f, T) ch->f = (T*)calloc((size_t)n + 1, sizeof(T))
    ALLOC(tok, int); ALLOC(lane, int); ALLOC(isq, int); ALLOC(valid, int); ALLOC(rank, int);
    ALLOC(gstart, int); ALLOC(gend, int); ALLOC(slot, int64_t); ALLOC(val, double); ALLOC(x, double);
    ALLOC(logv, double); ALLOC(rex, double); ALLOC(gtot, double); ALLOC(gabs, double);
    ALLOC(kb, int); ALLOC(ka, int); ALLOC(qb, int); ALLOC(qa, int); ALLOC(rep, int);
    ALLOC(order, int); ALLOC(ents, ent_t);
#undef ALLOC
    int bad = 0;
    for (int t = 0; t < C; ++t) {
        for (int j = 0; j < wr; ++j) {
            const int e = t * wr + j;
            const int q = j >= W;
            const int a = q ? j - W : j;
            const int64_t id = q ? (int64_t)q_idx[t * R + a] : (int64_t)k_idx[t * W + a];
            ch->tok[e] = t;
            ch->lane[e] = a;
            ch->isq[e] = q;
            ch->valid[e] = t < V;
            ch->val[e] = q ? q_val[t * R + a] : k_val[t * W + a];
            ch->slot[e] = id;
            if (ch->valid[e] && (id < 0 || id >= S)) bad = 1;
            /* invalid entries sort after every valid one, in index order */
            ch->ents[e].key = ch->valid[e] ? id : INT64_MAX;
            ch->ents[e].e = e;
        }
    }
    qsort(ch->ents, (size_t)n, sizeof(ent_t), cmp_ent);
    for (int r = 0; r < n; ++r) {
        ch->order[r] = ch->ents[r].e;
        ch->rank[ch->ents[r].e] = r;
    }
    /* Groups: maximal runs of one slot among valid entries; an invalid entry is its own group. */
    int r = 0;
    while (r < n) {
        const int e0 = ch->order[r];
        int r1 = r + 1;
        if (ch->valid[e0]) {
            while (r1 < n && ch->valid[ch->order[r1]] && ch->ents[r1].key == ch->ents[r].key) ++r1;
        }
        /* gates: a write entry, unless the entry before it in the group is a write entry of the
         * same token (that token has already decayed the slot) */
        double run = 0.0, tot = 0.0, tabs = 0.0;
        int nk = 0, nq = 0;
        for (int s = r; s < r1; ++s) {
            const int e = ch->order[s];
            double xe = 0.0;
            if (ch->valid[e] && !ch->isq[e]) {
                const int prev_same = s > r && !ch->isq[ch->order[s - 1]] && ch->valid[ch->order[s - 1]] &&
                                      ch->tok[ch->order[s - 1]] == ch->tok[e];
                ch->rep[e] = prev_same;
                if (!prev_same) xe = g[ch->tok[e] * g_width + ch->lane[e] * g_lane_stride];
            }
            ch->x[e] = xe;
            tot += xe;
            tabs += fabs(xe);
            if (ch->valid[e]) {
                if (ch->isq[e]) ++nq; else ++nk;
            }
        }
        int kseen = 0, qseen = 0;
        for (int s = r; s < r1; ++s) {
            const int e = ch->order[s];
            run += ch->x[e];
            ch->gstart[e] = r;
            ch->gend[e] = r1;
            ch->gtot[e] = tot;
            ch->gabs[e] = tabs;
            if (!ch->valid[e]) continue;
            ch->logv[e] = run;         /* inclusive: a read entry sees its own token's gate */
            double after = 0.0;
            for (int u = s + 1; u < r1; ++u) after += ch->x[ch->order[u]];
            ch->rex[e] = ch->isq[e] ? 0.0 : after;
            ch->kb[e] = kseen;
            ch->qb[e] = qseen;
            if (ch->isq[e]) ++qseen; else ++kseen;
            ch->ka[e] = nk - kseen;    /* after this entry (it counted itself above) */
            ch->qa[e] = nq - qseen;
        }
        r = r1;
    }
    return bad ? -1 : 0;
}

static uint32_t payload_bits(const chunk_t* ch, int e) {
    return (uint32_t)ch->tok[e] << 9 | (uint32_t)ch->isq[e] << 8 | (uint32_t)ch->lane[e] |
           (ch->valid[e] ? 0u : 0x20000u);
}

static int imin(int a, int b) { return a < b ? a : b; }

/* ---- Phase 1 ------------------------------------------------------------------------------- */

/*
 * Phase 1 of nchunks chunks (chunk c: tokens of the chunk valid when t < V, V = valid_last for
 * c >= first_partial, else C). Inputs are chunk-major: k_idx [nchunks, C, W], q_idx [.., C, R],
 * values as float64, g [nchunks, C] (g_per_entry = 0) or [nchunks, C, W] (1).
 * Outputs (entry order [nchunks, C, W] / [nchunks, C, R]; any pointer may be NULL):
 *   log_k, rex, cpe, k_eff, is_last, is_only, pos_k, gabs_k (sum |x| of the entry's group),
 *   log_q, q_w, pos_q, q_last, q_only, gabs_q,
 *   sorted_k [nchunks, C * W], sorted_q [nchunks, C * R] (the kinds' sorted rows),
 *   A, QK [nchunks, C, C] with A_abs, QK_abs = the sum of |term| per cell, repeats (one count).
 * Returns 0, or -1 if a valid slot id is out of range.
 */
int sdm_oracle_phase1(int64_t nchunks, int C, int W, int R, int64_t first_partial, int valid_last,
                      int g_per_entry, int64_t S, const int32_t* k_idx, const int32_t* q_idx,
                      const double* k_val, const double* q_val, const double* g, double* log_k,
                      double* rex, double* cpe, double* k_eff, int8_t* is_last, int8_t* is_only,
                      int32_t* pos_k, double* gabs_k, double* log_q, double* q_w, int32_t* pos_q,
                      int8_t* q_last, int8_t* q_only, double* gabs_q, int32_t* sorted_k,
                      int32_t* sorted_q, double* A, double* QK, double* A_abs, double* QK_abs,
                      int64_t* repeats) {
    const int wr = W + R;
    const int g_width = g_per_entry ? W : 1, g_ls = g_per_entry ? 1 : 0;
    int64_t reps = 0;
    int status = 0;
    for (int64_t c = 0; c < nchunks; ++c) {
        const int V = c >= first_partial ? valid_last : C;
        chunk_t ch;
        if (chunk_analyze(&ch, C, W, R, V, S, k_idx + c * C * W, q_idx + c * C * R, k_val + c * C * W,
                          q_val + c * C * R, g + c * C * g_width, g_width, g_ls) != 0)
            status = -1;
        const int64_t kw = c * C * W, qr = c * C * R;
        /* per-entry fields */
        for (int e = 0; e < ch.n; ++e) {
            const int t = ch.tok[e], a = ch.lane[e], v = ch.valid[e], r = ch.rank[e];
            const int after = ch.isq[e] ? ch.qa[e] : ch.ka[e];
            const int before = ch.isq[e] ? ch.qb[e] : ch.kb[e];
            const int asat = imin(after, 127);
            const uint32_t packed = v ? ((uint32_t)r | (uint32_t)asat << 17 |
                                         (uint32_t)imin(before + 1 + asat, 127) << 24)
                                      : (uint32_t)r;
            if (!ch.isq[e]) {
                const int64_t o = kw + t * W + a;
                reps += v && ch.rep[e];
                if (log_k) log_k[o] = v ? ch.logv[e] : 0.0;
                if (rex) rex[o] = v ? ch.rex[e] : 0.0;
                if (cpe) cpe[o] = v ? exp(ch.gtot[e]) : 1.0;
                if (k_eff) k_eff[o] = v ? ch.val[e] * exp(ch.logv[e]) : 0.0;
                if (is_last) is_last[o] = (int8_t)(v && after == 0);
                if (is_only) is_only[o] = (int8_t)(v && after == 0 && before == 0);
                if (pos_k) pos_k[o] = (int32_t)packed;
                if (gabs_k) gabs_k[o] = ch.gabs[e];
            } else {
                const int64_t o = qr + t * R + a;
                if (log_q) log_q[o] = v ? ch.logv[e] : 0.0;
                if (q_w) q_w[o] = v ? ch.val[e] * exp(ch.logv[e]) : 0.0;
                if (q_last) q_last[o] = (int8_t)(v && after == 0);
                if (q_only) q_only[o] = (int8_t)(v && after == 0 && before == 0);
                if (pos_q) pos_q[o] = (int32_t)packed;
                if (gabs_q) gabs_q[o] = ch.gabs[e];
            }
        }
        /* sorted rows of each kind: the kind's entries in sorted order */
        int jk = 0, jq = 0;
        for (int r = 0; r < ch.n; ++r) {
            const int e = ch.order[r];
            const int v = ch.valid[e];
            const int after = ch.isq[e] ? ch.qa[e] : ch.ka[e];
            const int before = ch.isq[e] ? ch.qb[e] : ch.kb[e];
            uint32_t el = payload_bits(&ch, e) & 0x3FFFFu;
            if (v) {
                el |= (uint32_t)imin(before, 4095) << 18;
                if (before == 0) el |= 0x80000000u;
                if (after == 0) el |= 0x40000000u;
            } else {
                el |= 0xC0000000u;
            }
            if (ch.isq[e]) {
                if (sorted_q) sorted_q[qr + jq] = (int32_t)el;
                ++jq;
            } else {
                if (sorted_k) sorted_k[kw + jk] = (int32_t)el;
                ++jk;
            }
        }
        /* pair triangles: per group, every valid entry e of token i with every valid write entry f
         * of token j in the same group; A (e a write entry) takes j < i, QK (e a read entry) j <= i */
        if (A || QK || A_abs || QK_abs) {
            const int64_t base = c * C * C;
            for (int i = 0; i < C * C; ++i) {
                if (A) A[base + i] = 0.0;
                if (QK) QK[base + i] = 0.0;
                if (A_abs) A_abs[base + i] = 0.0;
                if (QK_abs) QK_abs[base + i] = 0.0;
            }
            for (int r = 0; r < ch.n; ++r) {
                const int e = ch.order[r];
                if (!ch.valid[e]) continue;
                const int i = ch.tok[e];
                for (int s = ch.gstart[e]; s < ch.gend[e]; ++s) {
                    const int f = ch.order[s];
                    if (!ch.valid[f] || ch.isq[f]) continue;
                    const int j = ch.tok[f];
                    const double term = ch.val[e] * ch.val[f] * exp(ch.logv[e] - ch.logv[f]);
                    if (!ch.isq[e] && j < i) {
                        if (A) A[base + (int64_t)i * C + j] += term;
                        if (A_abs) A_abs[base + (int64_t)i * C + j] += fabs(term);
                    } else if (ch.isq[e] && j <= i) {
                        if (QK) QK[base + (int64_t)i * C + j] += term;
                        if (QK_abs) QK_abs[base + (int64_t)i * C + j] += fabs(term);
                    }
                }
            }
        }
        (void)wr;
        chunk_free(&ch);
    }
    if (repeats) *repeats = reps;
    return status;
}

/* ---- DW --------------------------------------------------------------------------------------- */

/*
 * Decay-and-write of ONE chunk into its stream's bank rows (bank [S, hd], float64, in place).
 * Per slot group with valid write entries: new = base * cpe_last + sum_m k_m exp(rex_m) dv[tok_m],
 * cpe_last = exp(group total) rounded to the value type when round_cpe (val_bf16 selects
 * bfloat16, else float32), and new rounded to the bank type when round_bank (bank_bf16).
 * dv: [C, hd] float64 rows of the chunk's tokens.
 * alt (nullable, [S, hd]): for a row whose cpe lies so near a rounding boundary of the value type
 * that float32 arithmetic may round it the other way, the row's value with the other rounding;
 * elsewhere the same value as bank. amb (nullable, [S]) counts such rows; touched ([S]) counts writes.
 * mag (nullable, [S, hd]): |base * cpe_last| + sum_m |sc_m * dv[tok_m]| of the row's last write, the
 * scale of the rounding error a float32 evaluation of the row can make.
 * Returns 0, or -1 if a valid slot id is out of range.
 */
int sdm_oracle_dw_chunk(int C, int W, int R, int V, int g_per_entry, int64_t S, int hd,
                        const int32_t* k_idx, const int32_t* q_idx, const double* k_val,
                        const double* q_val, const double* g, const double* dv, double* bank,
                        double* alt, int32_t* amb, int32_t* touched, double* mag, int round_cpe, int val_bf16,
                        int round_bank, int bank_bf16, double amb_rel) {
    const int g_width = g_per_entry ? W : 1, g_ls = g_per_entry ? 1 : 0;
    chunk_t ch;
    const int st = chunk_analyze(&ch, C, W, R, V, S, k_idx, q_idx, k_val, q_val, g, g_width, g_ls);
    double* acc = (double*)calloc((size_t)hd, sizeof(double));
    double* aabs = (double*)calloc((size_t)hd, sizeof(double));
    int r = 0;
    while (r < ch.n) {
        const int e0 = ch.order[r];
        const int r1 = ch.gend[e0];
        /* members: the group's valid write entries, in sorted order */
        int members = 0;
        for (int i = 0; i < hd; ++i) acc[i] = aabs[i] = 0.0;
        int64_t s = -1;
        for (int u = r; u < r1; ++u) {
            const int e = ch.order[u];
            if (!ch.valid[e] || ch.isq[e]) continue;
            const double sc = ch.val[e] * exp(ch.rex[e]);
            const double* row = dv + (int64_t)ch.tok[e] * hd;
            for (int i = 0; i < hd; ++i) {
                acc[i] += sc * row[i];
                aabs[i] += fabs(sc * row[i]);
            }
            s = ch.slot[e];
            ++members;
        }
        if (members > 0 && s >= 0 && s < S) {
            const double exact = exp(ch.gtot[e0]);
            const double cp = round_cpe ? round_to(exact, val_bf16) : exact;
            int ambiguous = 0;
            double cp_alt = cp;
            if (round_cpe && amb_rel > 0.0) {
                const double lo = round_to(exact * (1.0 - amb_rel), val_bf16);
                const double hi = round_to(exact * (1.0 + amb_rel), val_bf16);
                if (lo != hi) {
                    ambiguous = 1;
                    cp_alt = (cp == lo) ? hi : lo;
                }
            }
            double* brow = bank + s * hd;
            double* arow = alt ? alt + s * hd : NULL;
            for (int i = 0; i < hd; ++i) {
                const double base = brow[i];
                if (mag) mag[s * hd + i] = fabs(base * cp) + aabs[i];
                double nv = base * cp + acc[i];
                if (arow) {
                    /* an earlier ambiguity of this row carries on through its own alternative */
                    const double abase = (amb && amb[s]) ? arow[i] : base;
                    double av = abase * (ambiguous ? cp_alt : cp) + acc[i];
                    arow[i] = round_bank ? round_to(av, bank_bf16) : av;
                }
                brow[i] = round_bank ? round_to(nv, bank_bf16) : nv;
            }
            if (amb && ambiguous) amb[s] += 1;
            if (touched) touched[s] += 1;
        }
        r = r1;
    }
    free(acc);
    free(aabs);
    chunk_free(&ch);
    return st;
}
