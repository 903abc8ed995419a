/*
 * gdn.h — C ABI of the GB300 (sm_103a) Gated DeltaNet layer core.
 *
 * The library computes, on one GPU, the four pieces of the GDN layer core:
 *
 *   gdn_conv           width-W causal depthwise conv over the concatenated
 *                      q|k|v channels, then SiLU, with a rolling conv window
 *                      kept in each request's page;
 *   gdn_seq            the gated delta rule token by token (decode and short
 *                      prefill), q/k L2 norm and gates fused in;
 *   gdn_spec_verify    speculative-decode verify with ONE state page per
 *                      request: replay the accepted rows of the previous
 *                      step from the page's record, checkpoint the state,
 *                      run the new candidates (row count 0 = commit);
 *   gdn_chunk_prefill  the chunked (WY) form of the same rule for long
 *                      prompts, contractions on the tcgen05 tensor cores.
 *
 * Sources (the method is described, not printed, on these pages):
 *   - r9700-stack v0.2.4 release notes, "What it does": one state page per
 *     request holding the state, a two-slot record of the previous step's
 *     candidate rows (conv'd q/k/v and a/b gates) and a flag word (live
 *     slot, parity, done counter); replay, checkpoint, run candidates.
 *   - r9700-stack v0.2.4, "A defect found and fixed before the tag": the
 *     conv window rolls by the number of candidate columns, read from the
 *     record, never from the caller's tensor widths.
 *   - r9700-stack v0.2.3, section 1 "Time to first token: the GDN prefill
 *     core": token-by-token core (r9k_gdn_seq) and one-launch causal conv
 *     (r9k_gdn_conv) that address the batch's own rows through a row map;
 *     an fp64 token-by-token reference; the chunked core for long prompts.
 *   - vllm.cpp PR #155, "What changed": the post-conv q/k L2 norm and gate
 *     step fused per token; the width-4 causal conv specialisation.
 *   The rule itself: per value head with state S (Dk x Dv),
 *     g_t = -exp(A_log) softplus(a_t + dt_bias), beta_t = sigmoid(b_t),
 *     S <- e^{g_t} S, u = beta_t (v_t - S^T k_t), S <- S + k_t u^T,
 *     o_t = scale S^T q_t, with q_t, k_t L2-normalised.
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" point to GPU memory, "host" to CPU memory.
 *     The caller owns every buffer; the library allocates nothing and keeps
 *     no global state.
 *   - Every call is asynchronous on the given CUDA stream (0 = legacy
 *     default stream) and never synchronises. Kernels are launched with
 *     programmatic stream serialization and wait for the previous work on
 *     the stream before touching any memory, so ordering is that of plain
 *     launches; back-to-back calls overlap only their launch latency.
 *   - Host-side problems (null pointers, bad sizes, unsupported shapes) are
 *     returned as a negative gdn_status BEFORE anything is launched or
 *     written.
 *   - Per-request problems found on the device (bad page index, bad accepted
 *     count, stale step parity, ...) are written to *status (device int32)
 *     as a positive gdn_status: the first error wins (atomic compare-and-swap
 *     from 0), the offending request is skipped, the others complete. Callers
 *     zero *status before the call and read it when convenient. Kernels never
 *     trap.
 *   - Results for a request depend only on that request's inputs, never on
 *     the composition or order of the batch, and are run-to-run identical
 *     (no floating-point atomics anywhere).
 *
 * Layouts (row-major, innermost last)
 *   rows:    x, y (conv'd) [num_rows][C], C = 2*Hk*Dk + Hv*Dv, channel
 *            order [q (Hk x Dk) | k (Hk x Dk) | v (Hv x Dv)];
 *            a, b [num_rows][Hv]; o [num_rows][Hv][Dv].
 *   conv_w:  [C][W], io dtype.       A_log, dt_bias: [Hv] fp32.
 *   GQA:     value head h reads q/k head floor(h * Hk / Hv).
 *   page:    see gdn_page_layout(); the state inside a page is
 *            [Hv][Dv][Dk] (for each value column j, the Dk entries S[:, j]
 *            are contiguous).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdn_stream_t; /* same handle as cudaStream_t */

typedef enum {
  GDN_OK = 0,
  /* host-side, returned by the call (nothing launched, nothing written) */
  GDN_ERR_INVALID_ARG = -1,   /* null pointer, negative count, bad enum      */
  GDN_ERR_UNSUPPORTED = -2,   /* shape outside what the kernels support      */
  GDN_ERR_LAUNCH = -3,        /* the CUDA runtime refused a launch           */
  GDN_ERR_WORKSPACE = -4,     /* workspace smaller than required             */
  GDN_ERR_NO_DEVICE = -5,     /* no usable sm_100-family device / driver     */
  /* device-side, written to *status (first error wins; request skipped)     */
  GDN_DEV_BAD_PAGE = 1,       /* page index outside [0, num_pages)           */
  GDN_DEV_BAD_ROWS = 2,       /* row range outside [0, num_rows) / > max_rows */
  GDN_DEV_BAD_ACCEPTED = 3,   /* accepted count outside [0, record width)    */
  GDN_DEV_STALE_STEP = 4,     /* page parity differs from the request's bit  */
  GDN_DEV_TOO_MANY_CANDIDATES = 5, /* spec row count above max_candidates   */
  GDN_DEV_RECORD_OPEN = 6,    /* plain rows on a page with an open record    */
  GDN_DEV_BAD_FLAG = 7,       /* corrupt flag word, or FRESH with SPEC       */
  GDN_DEV_TIMEOUT = 8         /* a bounded on-chip wait gave up (the request's
                                 results are not written)                    */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Shapes and dtypes of one GDN layer. Supported: Dk = Dv in {32, 64, 128},
 * Hv a multiple of Hk, W = 4, 0 <= max_candidates <= 8. */
typedef struct {
  int32_t num_k_heads;     /* Hk: q/k heads                                 */
  int32_t num_v_heads;     /* Hv: value heads (= state heads)               */
  int32_t head_k_dim;      /* Dk                                             */
  int32_t head_v_dim;      /* Dv                                             */
  int32_t conv_width;      /* W                                              */
  int32_t max_candidates;  /* Kc: record rows per slot, 0 = no spec record   */
  int32_t io_dtype;        /* gdn_dtype of x, y, a, b, conv_w, window, record */
  int32_t state_dtype;     /* gdn_dtype of S in pages                        */
  int32_t out_dtype;       /* gdn_dtype of o                                 */
} gdn_dims;

/* Per-layer parameters. */
typedef struct {
  const float* A_log;      /* device [Hv]                                    */
  const float* dt_bias;    /* device [Hv]                                    */
  const float* conv_bias;  /* device [C] or NULL (no bias)                   */
  float scale;             /* output scale; <= 0 selects Dk^-1/2             */
  float norm_eps;          /* q/k L2 norm: x / sqrt(sum x^2 + norm_eps)      */
  int32_t gate_mode;       /* 0: a, b are raw (softplus/sigmoid in kernel);
                              1: a is g (log decay) and b is beta, given     */
} gdn_params;

/* Request flags (gdn_batch.flags). */
#define GDN_REQ_FRESH  0x1u  /* new sequence: zero state and conv window    */
#define GDN_REQ_SPEC   0x2u  /* rows are speculative candidates (verify)    */
#define GDN_REQ_PARITY 0x4u  /* expected step parity of a SPEC page         */

/* The row map of one step: which packed rows belong to which request and
 * page. All arrays are device memory with num_requests entries. */
typedef struct {
  int32_t num_requests;       /* R                                           */
  int32_t num_rows;           /* rows in the packed x/y/a/b/o buffers        */
  int32_t max_rows;           /* upper bound on any row_len (host-known)     */
  int32_t num_pages;          /* pages in the pool (page index bound)        */
  const int32_t* row_start;   /* device [R]: first packed row of request r   */
  const int32_t* row_len;     /* device [R]: rows of request r this step     */
  const int32_t* page;        /* device [R]: page index of request r         */
  const uint32_t* flags;      /* device [R]: GDN_REQ_* bits                  */
  const int32_t* n_accepted;  /* device [R]: SPEC: drafts accepted by the
                                 previous step (rows 0..n_accepted replayed);
                                 may be NULL when no request is SPEC         */
  const int32_t* order;       /* device [R] or NULL: processing order, e.g.
                                 longest first (a permutation of 0..R-1)     */
} gdn_batch;

/* Byte layout of one state page (all offsets 256-byte aligned).
 *   window  [(W-1) + Kc][C] io dtype: conv window. Columns 0..W-2 hold the
 *           last W-1 raw input columns before the record's candidates;
 *           columns W-1.. hold the raw candidate columns of the live record.
 *   state   [Hv][Dv][Dk] state dtype: the GDN state (the checkpoint).
 *   record  [2][Kc][R_w] io dtype: two slots of candidate rows, each row
 *           = conv'd q|k|v (C) then a (Hv) then b (Hv), padded to R_w
 *           elements so that every row starts on a 16-byte boundary; then
 *           [2][Hv][216] fp32: per slot and value head, the run coefficients
 *           the verify derived for that slot's rows (G_t [8] and
 *           R[t][s]/|k_s| [8][8], which the next step's replay uses as
 *           stored; then G_t/|k_t| [8], G_t/|q_t| [8], M = (I - L)^-1
 *           diag(beta) [8][8] and N [8][8]; see gdn_spec_verify); then
 *           [Hv][Kc][Dv] fp32: the live slot's u_t per value column, which
 *           the next step's replay applies as stored (and then overwrites
 *           with its own candidates' u).
 *   flag    uint32: bit 0 live slot, bit 1 step parity, bits 2..7 number of
 *           rows in the live slot, bits 8..31 done counter (0 between calls).
 * A zero-filled page is a valid empty page (zero state, zero window, closed
 * record, parity 0). */
typedef struct {
  size_t page_bytes;
  size_t window_offset, window_bytes;
  size_t state_offset, state_bytes;
  size_t record_offset, record_bytes;
  size_t flag_offset;
} gdn_page_layout_t;

/* Page layout for these dims. Host only; launches nothing. */
gdn_status gdn_page_layout(const gdn_dims* dims, gdn_page_layout_t* out);

/* Causal conv + SiLU over the step's rows (r9700-stack v0.2.3, section 1:
 * r9k_gdn_conv; v0.2.4: window width from the record).
 *   y_t[c] = SiLU( bias[c] + sum_{j=0..W-1} w[c][j] * x_{t-(W-1)+j}[c] )
 * accumulated in fp32 in exactly that order (fused multiply-adds, taps
 * oldest first), SiLU(z) = z / (1 + e^{-z}) = z sigmoid(z), evaluated from
 * the library's own exp of -|z| and the correctly rounded quotient
 * e^{-|z|} / (1 + e^{-|z|}) (each step one rounding of a plain operation, so
 * a plain CPU program reproduces every output bit; within 4 ulp of the
 * exact value).
 * History before a request's first row comes from its page window (zero for
 * FRESH requests). Per request:
 *   plain:  window columns 0..W-2 <- last W-1 columns of [history; rows];
 *           the page's record must be closed (else GDN_DEV_RECORD_OPEN).
 *   SPEC:   history = window columns a+1..a+W-1 where a = n_accepted (or
 *           0..W-2 when the record is empty); then window columns 0..W-2 <-
 *           history, columns W-1.. <- this step's raw candidates, and the
 *           conv'd candidate rows are also written to record slot 1-live.
 *           row_len <= max_candidates.
 *   x       device [num_rows][C] io dtype (raw conv inputs)
 *   conv_w  device [C][W] io dtype
 *   y       device [num_rows][C], dtype y_dtype (GDN_F32 or the io dtype)
 *   pages   device page pool (gdn_page_layout().page_bytes each)
 *   status  device int32 (see conventions)                                */
gdn_status gdn_conv(const gdn_dims* dims, const gdn_batch* batch,
                    const gdn_params* params, const void* x, const void* conv_w,
                    void* y, int32_t y_dtype, void* pages, int32_t* status,
                    gdn_stream_t stream);

/* Token-by-token gated delta rule for the plain (non-SPEC) requests of the
 * batch; SPEC requests are skipped (r9700-stack v0.2.3, section 1:
 * r9k_gdn_seq, any number of tokens, state in registers). Per request the
 * state is read from its page (zero if FRESH), each row t computes
 *   q^ = q/sqrt(|q|^2+eps), k^ likewise, g, beta from a, b (gate_mode),
 *   S <- e^g S; u = beta (v - S^T k^); S <- S + k^ u^T; o = scale S^T q^
 * and the final state is written back to the page. A FRESH request also
 * resets the page's flag word to an empty record.
 *   qkv  device [num_rows][C] io dtype (conv'd rows, i.e. gdn_conv's y)
 *   a, b device [num_rows][Hv] io dtype;  o device [num_rows][Hv][Dv]      */
gdn_status gdn_seq(const gdn_dims* dims, const gdn_batch* batch,
                   const gdn_params* params, const void* qkv, const void* a,
                   const void* b, void* o, void* pages, int32_t* status,
                   gdn_stream_t stream);

/* Fused decode step: gdn_conv (io-dtype output) followed by gdn_seq for a
 * batch of one token per request, in one launch, with the same results bit
 * for bit (outputs, states, conv windows; the conv'd rows are not written).
 * This is the "one launch per layer" design the r9700-stack v0.2.3 notes
 * (section 1) credit for the short-step speed-up, extended to the conv.
 * Plain requests with row_len 1 (or 0: a FRESH request is zeroed) are
 * processed; SPEC requests are skipped; row_len > 1 is GDN_DEV_BAD_ROWS.
 * Requires (Hv/Hk) * (Dv/32) <= 16 and batch->max_rows <= 1.
 *   x       device [num_rows][C] io dtype (raw conv inputs)
 *   conv_w  device [C][W];  a, b, o, pages, status as gdn_seq.            */
gdn_status gdn_decode(const gdn_dims* dims, const gdn_batch* batch,
                      const gdn_params* params, const void* x,
                      const void* conv_w, const void* a, const void* b,
                      void* o, void* pages, int32_t* status,
                      gdn_stream_t stream);

/* One-page speculative verify for the SPEC requests of the batch; plain
 * requests are skipped (r9700-stack v0.2.4, "What it does";
 * r9k_gdn_spec_verify / r9k_gdn_spec_commit). Per SPEC request with page
 * flag (live slot L, parity P, width n):
 *   1. P must equal the request's GDN_REQ_PARITY bit (else
 *      GDN_DEV_STALE_STEP, request untouched);
 *   2. if n > 0: replay rows 0..a (a = n_accepted, 0 <= a < n) of record
 *      slot L into the page state and store it (the new checkpoint): the
 *      rank-(a+1) update with the rows' G, R/|k| and u as the previous step
 *      stored them;
 *   3. run this step's row_len candidates (qkv rows, a, b) from the
 *      checkpoint, writing o for each; no per-candidate state is kept;
 *   4. write the candidates' a/b into record slot 1-L (gdn_conv wrote their
 *      conv'd rows there);
 *   5. the last block to finish sets L <- 1-L (if row_len > 0), n <-
 *      row_len, P <- 1-P, counter <- 0.
 * row_len == 0 is the commit: replay, checkpoint, close the record.
 * Arguments as gdn_seq. Bit-identical to gdn_spec_slots on the same rows.
 * Each run of rows (the replay, then the candidates) is evaluated in closed
 * form from the state it starts at: with decay products R[t][s] =
 * e^{g_{s+1}} ... e^{g_t} and G_t = e^{g_0} ... e^{g_t},
 *   u_t = beta_t (v_t - G_t S^T k^_t - sum_{s<t} R[t][s] (k^_s.k^_t) u_s),
 *   o_t = scale (G_t S^T q^_t + sum_{s<=t} R[t][s] (k^_s.q^_t) u_s),
 *   checkpoint S_a = G_a S + sum_{s<=a} R[a][s] k^_s u_s^T,
 * which equals the token-by-token rule in exact arithmetic. Two launches on
 * `stream`: the candidates' coefficients per (request, q/k head), written to
 * record slot 1-L, then the items per (request, value head), which also
 * store the candidates' u for the next step. Returns GDN_ERR_UNSUPPORTED
 * when a q/k head's group of value heads is too wide for the kernels'
 * shared memory (more than 124 value heads per q/k head at Dk = Dv = 128
 * with bf16 rows and fp32 state). */
gdn_status gdn_spec_verify(const gdn_dims* dims, const gdn_batch* batch,
                           const gdn_params* params, const void* qkv,
                           const void* a, const void* b, void* o, void* pages,
                           int32_t* status, gdn_stream_t stream);

/* Fused speculative step: gdn_conv (io-dtype output) followed by
 * gdn_spec_verify for the SPEC requests of the batch, without a separate
 * conv launch, with the same results bit for bit (outputs, states, conv
 * windows, record slots and flag words; the conv'd rows are written only
 * into the record, as the next step's replay needs them). Plain requests
 * are skipped. This is the fewer-launches-per-layer-step design that the
 * r9700-stack v0.2.3 notes (section 1) credit for the short-step speed-up,
 * applied to the verify of v0.2.4 ("What it does"): one launch, one CTA
 * per (request, q/k head), which convolves the group's q, k and v channels
 * for this step's candidates and rolls the window by the accepted count,
 * forms the group's run coefficients, then replays, checkpoints and runs the
 * candidates for every value column of the group. One launch, against three
 * for gdn_conv + gdn_spec_verify.
 *   x       device [num_rows][C] io dtype (raw conv inputs, candidate rows)
 *   conv_w  device [C][W];  a, b, o, pages, status as gdn_spec_verify.
 * Returns GDN_ERR_UNSUPPORTED when the group's rows and replay u do not fit
 * in shared memory (more than 18 value heads per q/k head at Dk = Dv = 128
 * with bf16 rows and fp32 state; gdn_conv + gdn_spec_verify take such
 * shapes). */
gdn_status gdn_spec_step(const gdn_dims* dims, const gdn_batch* batch,
                         const gdn_params* params, const void* x,
                         const void* conv_w, const void* a, const void* b,
                         void* o, void* pages, int32_t* status,
                         gdn_stream_t stream);

/* Slot-per-candidate speculative decode: the stock layout the one-page
 * verify replaces (r9700-stack v0.2.4, "What it does": a state page per
 * candidate, 1 + 7 per request). Request r owns the slot pool at byte
 * page[r] * pool_bytes of `slots` (gdn_slot_layout); slot i holds a state
 * [Hv][Dv][Dk] (state dtype) and a conv window [W-1][C] (io dtype). The call
 * resumes request r from slot n_accepted[r] (0 <= n_accepted < Kc; the
 * caller seeds slot 0 before the first step), runs its row_len candidates
 * through conv and rule, and stores the state and window after candidate i
 * into slot i. Two launches (conv, then the closed-form run per candidate)
 * on `stream`. Returns GDN_ERR_UNSUPPORTED when the group's rows do not fit
 * in shared memory (more than 42 value heads per q/k head at Dk = Dv = 128
 * with bf16 rows and fp32 state).
 *   x     device [num_rows][C] raw candidate rows (io dtype)
 *   y     device [num_rows][C] io dtype, receives the conv'd rows
 *   a, b, o, conv_w, status as gdn_conv / gdn_seq.                       */
typedef struct {
  size_t pool_bytes;     /* bytes per request (per page index)             */
  size_t slot_bytes;     /* stride between slots inside a pool             */
  size_t state_offset;   /* state of slot i at i*slot_bytes + state_offset */
  size_t window_offset;  /* window of slot i at i*slot_bytes + window_offset */
} gdn_slot_layout_t;

gdn_status gdn_slot_layout(const gdn_dims* dims, gdn_slot_layout_t* out);

gdn_status gdn_spec_slots(const gdn_dims* dims, const gdn_batch* batch,
                          const gdn_params* params, const void* x,
                          const void* conv_w, void* y, const void* a,
                          const void* b, void* o, void* slots,
                          int32_t* status, gdn_stream_t stream);

/* Hand a request between the one-page layout and the slot layout. The
 * r9700-stack v0.2.4 notes ("What it does") keep the stock per-candidate
 * pages when prefix caching is on, so a request may move from its state page
 * to a slot pool, or back, between steps. What moves is what the next step
 * starts from: the state and the W-1 history columns of the conv window.
 *
 * gdn_page_to_slots: for i < n, copies page page[i] (of `pages`, num_pages
 * pages) into slot 0 of slot pool pool[i] (of `slots`, num_pools pools); the
 * next gdn_spec_slots step of the request resumes from slot 0 (n_accepted 0).
 * The page's record must be closed (commit first, gdn_spec_verify with zero
 * rows), else the request is skipped with GDN_DEV_RECORD_OPEN.
 * gdn_slots_to_page: copies slot slot[i] (0 <= slot < max_candidates, e.g.
 * the accepted candidate) of pool pool[i] into page page[i] and closes the
 * page's record (empty record, step parity 0), so the next gdn_conv +
 * gdn_spec_verify of the request runs with GDN_REQ_PARITY clear.
 * page, pool, slot: device int32 [n]. Other device errors: GDN_DEV_BAD_PAGE
 * (an index out of range), GDN_DEV_BAD_ACCEPTED (a slot out of range); the
 * request is skipped. Requires max_candidates > 0 (else
 * GDN_ERR_UNSUPPORTED) and n <= 65535. One launch on `stream`. */
gdn_status gdn_page_to_slots(const gdn_dims* dims, int32_t n, const int32_t* page,
                             const int32_t* pool, int32_t num_pages, int32_t num_pools,
                             const void* pages, void* slots, int32_t* status,
                             gdn_stream_t stream);
gdn_status gdn_slots_to_page(const gdn_dims* dims, int32_t n, const int32_t* pool,
                             const int32_t* slot, const int32_t* page, int32_t num_pools,
                             int32_t num_pages, const void* slots, void* pages,
                             int32_t* status, gdn_stream_t stream);

/* Workspace bytes gdn_chunk_prefill needs for its two-pass form on this
 * batch (host only): num_requests x num_v_heads x ceil(max_rows / 64) items
 * of 99328 bytes (97 KiB). 0 when the chunked form does not support the
 * shape (io dtype other than bf16, Dk or Dv other than 128). */
size_t gdn_chunk_prefill_workspace_bytes(const gdn_dims* dims,
                                         const gdn_batch* batch);

/* Chunked prefill: the same rule as gdn_seq for the plain requests of the
 * batch, computed 64 tokens at a time in the WY (UT-transform) form
 * (r9700-stack v0.2.3, section 1, names the chunked core for prompts above
 * the token-by-token threshold). Per chunk with state S, gamma the in-chunk
 * prefix sums of g:
 *   A = strictly_lower(beta_t e^{gamma_t-gamma_s} k^_t.k^_s), T = (I+A)^-1,
 *   U = T diag(beta) V,  Wm = T diag(beta e^gamma) K^,  Vn = U - Wm S,
 *   O = scale (diag(e^gamma) Q^ S + (Q^ K^T o e^{gamma_t-gamma_s} o causal) Vn),
 *   S <- e^{gamma_L} S + (diag(e^{gamma_L-gamma}) K^)^T Vn.
 * Equal to gdn_seq in exact arithmetic; within 1e-4 relative in fp32.
 * Arguments as gdn_seq, plus a device workspace:
 *   workspace        NULL, or device memory of at least
 *                    gdn_chunk_prefill_workspace_bytes() bytes, 16-byte
 *                    aligned (else GDN_ERR_WORKSPACE / GDN_ERR_INVALID_ARG);
 *                    owned by the caller, overwritten, and in use until the
 *                    launches on `stream` complete.
 * With a workspace the call makes two launches. A pre-pass with one CTA per
 * (request, value head, chunk) does the steps that do not read the state
 * (the Gram products, A and its inverse T, U, Wm and the masked product P)
 * and stores Wm, U, P and the chunk's decay factors in the workspace; then
 * one CTA per (request, value head) walks the request's chunks with the
 * fp32 state in its tensor memory and does the rest (Wm S, Q^ S, P Vn and
 * the state update). With workspace NULL one launch does all of it on the
 * per-request chain. The two forms agree bit for bit. SPEC requests are
 * skipped. Requires io dtype bf16 and Dk = Dv = 128 (else
 * GDN_ERR_UNSUPPORTED) and qkv 16-byte aligned (the rows are read by TMA). */
gdn_status gdn_chunk_prefill(const gdn_dims* dims, const gdn_batch* batch,
                             const gdn_params* params, const void* qkv,
                             const void* a, const void* b, void* o,
                             void* pages, void* workspace,
                             size_t workspace_bytes, int32_t* status,
                             gdn_stream_t stream);

/* gdn_chunk_prefill's two-pass form with no caller workspace and no
 * allocation, for callers that cannot call cudaMalloc. The paper has no
 * counterpart: this is a deployment variant of gdn_chunk_prefill.
 * The workspace is a 64 MiB (67,108,864-byte) array in the library's device
 * image, one per device, held from the first use on that device until the
 * process exits. The first call on each device looks its address up
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before capturing a stream into a CUDA graph. Batches whose
 * gdn_chunk_prefill_workspace_bytes() exceed 64 MiB are rejected with
 * GDN_ERR_WORKSPACE (about 670 items of (request, value head, 64-row
 * chunk)). Every call shares the array and leaves its contents behind;
 * nothing in it needs to start at zero (the pre-pass of a call writes every
 * item that call reads). Calls whose launches overlap on the GPU (on
 * different streams, or from different threads) race on the array: order
 * them on one stream. Arguments, results and errors otherwise as
 * gdn_chunk_prefill with a workspace; GDN_ERR_LAUNCH also when the address
 * lookup fails. Calls no allocating routine.                                */
gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* dims, const gdn_batch* batch,
                                     const gdn_params* params, const void* qkv,
                                     const void* a, const void* b, void* o,
                                     void* pages, int32_t* status,
                                     gdn_stream_t stream);

/* Default row count from which gdn_prefill uses the chunked form. Measured on
 * GB300 (16/32 heads, Dk = Dv = 128): with 8 requests per step the chunked
 * form is faster from 32 rows (2.0x at 64, 2.7x at 1024); with a single
 * request from 64 rows (1.4x at 128, 1.6x at 1024). */
#define GDN_PREFILL_CHUNK_MIN_ROWS 64

/* Prefill dispatch: the plain requests of the batch with at least
 * chunk_min_rows rows (<= 0 selects GDN_PREFILL_CHUNK_MIN_ROWS) go through
 * gdn_chunk_prefill, the others through gdn_seq, each launch leaving the
 * other's requests alone. workspace / workspace_bytes as for
 * gdn_chunk_prefill on the same batch: with a workspace the chunked
 * requests take the two-pass form (three launches on `stream` in all),
 * with NULL the one-launch form (two launches). The r9700-stack v0.2.3 notes
 * (section 1) describe the same split by prefill length (R9K_GDN_PREFILL_MAX,
 * break-even measured per model and card); here the threshold is a call
 * argument. When the chunked form does not support the shape (io dtype other
 * than bf16, Dk or Dv other than 128, or an unaligned qkv) every request goes
 * token by token. Arguments otherwise as gdn_seq; SPEC requests are skipped. */
gdn_status gdn_prefill(const gdn_dims* dims, const gdn_batch* batch,
                       const gdn_params* params, const void* qkv, const void* a,
                       const void* b, void* o, void* pages,
                       int32_t chunk_min_rows, void* workspace,
                       size_t workspace_bytes, int32_t* status,
                       gdn_stream_t stream);

/* Failure-detection check of the bounded on-chip waits. Every wait a
 * kernel makes on its own bulk copies or MMAs (gdn_decode,
 * gdn_chunk_prefill) gives up after one second of global time: the kernel
 * then writes GDN_DEV_TIMEOUT to *status, lets its copies in flight land,
 * frees its tensor memory and returns, so the context stays usable. This
 * call runs that path on demand: one block waits on an mbarrier that
 * nothing arrives at, gives up after limit_ns of global time
 * (0 < limit_ns <= 10^10) and writes GDN_DEV_TIMEOUT to *status.
 *   status  device int32 (first error wins, as for every entry point)
 * Returns GDN_ERR_INVALID_ARG for a NULL status or a limit out of range. */
gdn_status gdn_check_bounded_wait(int64_t limit_ns, int32_t* status,
                                  gdn_stream_t stream);

/* Text for a status code (host, static storage). */
const char* gdn_strerror(int32_t status);

/* ABI version of this header: (major << 16) | minor. */
int32_t gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
