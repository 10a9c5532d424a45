/*
 * sdcp.h - C ABI of libsdcp, the batched acceptance step of a speculative-decoding
 * verifier, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the verifier's "Acceptance" step of the Speculative Decoding
 * Coordination Protocol (IETF draft-li-mlc-inference-acceleration-00, "Speculative
 * Decoding Coordination Protocol (SDCP) for Distributed Inference with Multi-Level
 * Caches"):
 *   - the sampling profile of Section 4.1 (temperature, then top-k, then top-p; a
 *     temperature of zero selects the most probable token, ties to the smallest id)
 *     turns logits into the distributions p (target) and q (draft);
 *   - Section 6.4, Rule 1 (greedy) and Rule 2 (speculative sampling) decide how many
 *     of the M proposed tokens are accepted and which one additional token is emitted;
 *   - Section 6.3, "Preconditions of the rule": q[i](x[i]) must be non-zero at every
 *     proposed position before any random value is drawn;
 *   - Section 6.3, "Scoring": the verifier may batch the proposals of many sessions;
 *   - Section 5.2, "verdict": the results are the accepted count a (0 <= a <= M) and
 *     the emitted tokens;
 *   - Table 2 (Section 6.9), problem types: a per-session status mirrors the ones that
 *     can arise inside this call.
 *
 * Random values are Philox4x32-10 uniforms (Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11), keyed by the session's
 * 64-bit seed (key word 0 = low 32 bits, key word 1 = high 32 bits), with counter
 * (position, purpose, round, session_tag); purpose 0 is the acceptance test and 1 the
 * additional token, as in SDCP Section 6.4.  The uniform is
 * ((w0 << 21) | (w1 >> 11)) * 2^-53, the first 53 bits of the output, like the
 * 53-bit value of Section 6.4.
 *
 * Ragged batch layout (all device memory, row-major, row stride V elements):
 *   B sessions; session b proposes M_b = m_offsets[b+1] - m_offsets[b] tokens.
 *   target row of session b at position i (i = 0..M_b):  T[m_offsets[b] + b + i]
 *   draft row of session b at position i (i = 0..M_b-1): D[m_offsets[b] + i]
 *   draft token of session b at position i:               draft_tokens[m_offsets[b] + i]
 *   output tokens of session b:                           out_tokens[m_offsets[b] + b + j],
 *                                                         j = 0..n_out[b]-1; the slots
 *                                                         j = n_out[b]..M_b hold -1.
 *
 * Ownership: the caller owns every buffer and the stream.  The library allocates
 * nothing, never synchronises the stream and keeps no state between calls, so calls on
 * different streams with different workspaces may run concurrently.  Results are a
 * pure function of the inputs: re-running a call reproduces every output bit for bit.
 *
 * Errors: a non-zero return code (SDCP_E_*) means nothing was launched (argument
 * errors) or a launch failed (SDCP_E_LAUNCH).  Errors that depend on values stored in
 * device memory are reported per session in status[] (SDCP_S_*); such a session gets
 * accepted = 0, n_out = 0 and all its output slots -1, and so commits nothing.
 */
#ifndef SDCP_H
#define SDCP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element types of the logits ------------------------------------------------ */
#define SDCP_F32  0   /* IEEE binary32 */
#define SDCP_BF16 1   /* bfloat16 (upper half of a binary32) */

/* ---- acceptance rules: SDCP Section 10.2.2 registry ------------------------------ */
#define SDCP_RULE_GREEDY 1              /* Rule 1 */
#define SDCP_RULE_SPECULATIVE_SAMPLING 2 /* Rule 2 */
/* A private-use rule (Section 10.2 keeps ids 192-255 for private use): the relaxed rule of
 * "Inference: KV Cache, Batching, Speculative Decoding" (section on variants of the
 * acceptance rule: accept if the token is in the target's top-k).  Acceptance test: x[i]
 * lies in the kept set of p[i], the target distribution after the session's sampling profile
 * (top_k = k makes it "in the target's top-k"), with a finite logit.  Additional token: a
 * draw from p[a] (purpose 1) at the first rejection, or from p[M+1] when all M are accepted;
 * argmax at temperature 0.  The proposal carries tokens only: draft rows are never read.  It
 * does NOT preserve the target distribution, and needs no trust in a drafter's q. */
#define SDCP_RULE_RELAXED_TOP_K 192

/* ---- return codes ---------------------------------------------------------------- */
#define SDCP_OK           0
#define SDCP_E_INVALID    1  /* null pointer, B < 0, V < 1, unknown dtype, sizes overflow */
#define SDCP_E_WORKSPACE  2  /* workspace null, too small or not 256-byte aligned */
#define SDCP_E_ALIGN      3  /* a logits pointer is not aligned to its element size */
#define SDCP_E_TOO_LARGE  4  /* V above SDCP_MAX_VOCAB or a row count above INT32_MAX */
#define SDCP_E_LAUNCH     5  /* a CUDA launch failed (cudaGetLastError after launch) */
#define SDCP_E_DEVICE     6  /* no usable CUDA device / device query failed */
#define SDCP_E_SCRATCH_LIMIT 7 /* batch needs more scratch than SDCP_NOALLOC_SCRATCH_BYTES */

/* ---- per-session status (mirrors SDCP Table 2 problem types) ---------------------- */
#define SDCP_S_OK             0
#define SDCP_S_BAD_PROPOSAL   1  /* "sdcp-bad-proposal": a token outside [0,V), or, under
                                    Rule 2, q[i](x[i]) = 0 at some position (Section 6.4) */
#define SDCP_S_LIMIT          2  /* "sdcp-limit": M outside [1, SDCP_MAX_M] (m_max <= 64,
                                    Section 4.1; 1 <= M, Section 6.2) */
#define SDCP_S_BAD_PARAMS     3  /* unknown rule id, top_p_milli > 1000, inconsistent
                                    m_offsets, or a scored row holding NaN, +inf or only
                                    -inf (no distribution can be formed) */
#define SDCP_S_Q_UNAVAILABLE  4  /* "sdcp-q-unavailable": Rule 2 without draft logits */
#define SDCP_S_INTERNAL       5  /* the call gave up a bounded wait on the GPU (a bulk copy
                                    that never completed); no output of the call is valid */

#define SDCP_MAX_M      64          /* m_max upper bound, SDCP Section 4.1 contract */
#define SDCP_MAX_VOCAB  (1 << 24)   /* ids and ranks are int32; 16 Mi keeps all sums exact */

/* One per session, device memory, 32 bytes, naturally aligned. */
typedef struct sdcp_session_params {
  uint32_t rule_id;           /* SDCP_RULE_*; anything else -> SDCP_S_BAD_PARAMS */
  uint32_t temperature_milli; /* temperature x 1000 (Section 4.1); 0 selects the argmax */
  uint32_t top_k;             /* keep the top_k most probable; 0 or >= V disables */
  uint32_t top_p_milli;       /* nucleus mass x 1000, <= 1000; 1000 disables */
  uint64_t seed;              /* Philox key of the verifier's random values */
  uint32_t round;             /* protocol round of this proposal */
  uint32_t session_tag;       /* 32 bits that name the session (e.g. the first four
                                 octets of its 16-octet identifier), not the batch slot */
} sdcp_session_params;

/*
 * Bytes of device workspace sdcp_verify_batch and sdcp_row_stats need for a batch of
 * B sessions with total_drafts = sum of M_b proposed tokens.  Returns 0 for invalid
 * sizes (B < 0, total_drafts < 0, V < 1 or V > SDCP_MAX_VOCAB).
 */
size_t sdcp_workspace_bytes(int64_t V, int32_t B, int64_t total_drafts);

/*
 * Verify one ragged batch (SDCP Sections 4.1, 6.3 and 6.4).
 *
 * target_logits  device, [total_drafts + B][V] of dtype; the scores p[1..M+1] of each
 *                session (Section 6.3 "Scoring"), laid out as described above.
 * draft_logits   device, [total_drafts][V] of dtype, or NULL when no session uses Rule 2
 *                (a Rule 2 session then gets SDCP_S_Q_UNAVAILABLE).  Rows of Rule 1
 *                sessions are never read.  The profile of the session is applied to these
 *                logits to form q (the draft distribution the tokens were sampled from).
 * dtype          SDCP_F32 or SDCP_BF16, for both logits arrays.
 * V              vocabulary size, 1..SDCP_MAX_VOCAB.  Any V is accepted; rows whose start
 *                is not 16-byte aligned are read with narrower loads at their ends.
 * B              number of sessions, >= 0 (B = 0 launches nothing).
 * m_offsets      device, [B+1] int32, m_offsets[0] = 0, non-decreasing,
 *                m_offsets[B] = total_drafts.  A session whose own pair m_offsets[b],
 *                m_offsets[b+1] is out of order or out of range gets SDCP_S_BAD_PARAMS;
 *                offsets out of order elsewhere leave the results of the sessions they
 *                overlap unspecified.  Never an out-of-range access.
 * total_drafts   host copy of m_offsets[B] (sizes the launch without a device read).
 * draft_tokens   device, [total_drafts] int32, the proposed tokens x[i].
 * params         device, [B] sdcp_session_params.
 * accepted       device out, [B] int32: a, the number of accepted draft tokens.
 * n_out          device out, [B] int32: a + 1 emitted tokens (0 for a failed session).
 * out_tokens     device out, [total_drafts + B] int32 (layout above).
 * status         device out, [B] int32 SDCP_S_*.
 * workspace      device scratch of at least sdcp_workspace_bytes(V, B, total_drafts)
 *                bytes, 256-byte aligned; its contents need no initialisation and are
 *                garbage afterwards.
 * stream         the cudaStream_t (as void*) all work is enqueued on; NULL = legacy stream.
 *
 * Returns SDCP_OK or SDCP_E_*.  Asynchronous: results are ready when the stream reaches
 * this point.
 */
int sdcp_verify_batch(const void* target_logits, const void* draft_logits, int dtype,
                      int64_t V, int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                      const int32_t* draft_tokens, const sdcp_session_params* params,
                      int32_t* accepted, int32_t* n_out, int32_t* out_tokens,
                      int32_t* status, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * The two phases of sdcp_verify_batch as separate calls (same arguments, same workspace):
 * phase 1 (sdcp_verify_rows) computes the statistics of every scored row of the sampling
 * profile (Section 4.1) into the workspace; phase 2 (sdcp_verify_sessions) runs the
 * precondition, the acceptance tests, the first-rejection scan and the draw of the
 * additional token (Sections 6.3, 6.4) and writes the outputs.  Calling phase 1 then
 * phase 2 on one stream is exactly sdcp_verify_batch; a profiler or a scheduler can put an
 * event between them.  Return codes as for sdcp_verify_batch.
 */
int sdcp_verify_rows(const void* target_logits, const void* draft_logits, int dtype,
                     int64_t V, int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                     const int32_t* draft_tokens, const sdcp_session_params* params,
                     void* workspace, size_t workspace_bytes, void* stream);
int sdcp_verify_sessions(const void* target_logits, const void* draft_logits, int dtype,
                         int64_t V, int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                         const int32_t* draft_tokens, const sdcp_session_params* params,
                         int32_t* accepted, int32_t* n_out, int32_t* out_tokens,
                         int32_t* status, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Per-row statistics of the sampling profile (parity hook for the first phase).
 *
 * Same inputs as sdcp_verify_batch.  For every target row r (0 <= r < total_drafts + B)
 * and then every draft row (total_drafts of them) it writes one sdcp_row_stat to
 * stats_out (device, [2 * total_drafts + B]), target rows first.  All rows are given the
 * full statistics regardless of the session's rule (draft rows of a session with an
 * invalid rule or M get flags = SDCP_ROW_SKIPPED).  Row statistics follow Section 4.1:
 *   lmax    the largest logit of the row (before temperature);
 *   log_s   natural log of S = sum over the kept set of exp((l_j - lmax) * 1000/T);
 *   lp_x    natural log of the probability of the row's draft token x (target row i < M
 *           and draft row i carry x[i]); -inf when x is outside the kept set or its
 *           logit is -inf; NaN for rows without a draft token (target row M) or x out
 *           of range;
 *   argmax  smallest id among the largest logits;
 *   kept    number of tokens in the kept set (1 when the temperature is 0);
 *   flags   SDCP_ROW_* bits.
 */
typedef struct sdcp_row_stat {
  float lmax;
  float log_s;
  float lp_x;
  int32_t argmax;
  int32_t kept;
  uint32_t thr_key;   /* internal: order key of the lowest kept value */
  int32_t thr_n;      /* internal: how many tokens with that value are kept, the first ones
                         in id order (INT32_MAX: all) */
  uint32_t flags;
} sdcp_row_stat;

#define SDCP_ROW_INVALID   1u  /* NaN, +inf, or no finite logit: no distribution */
#define SDCP_ROW_X_KEPT    2u  /* the draft token is in the kept set with a finite logit */
#define SDCP_ROW_SKIPPED   4u  /* row not processed */
#define SDCP_ROW_FALLBACK  8u  /* the threshold needed the generic multi-pass search */

int sdcp_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                   int64_t V, int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                   const int32_t* draft_tokens, const sdcp_session_params* params,
                   sdcp_row_stat* stats_out, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * sdcp_verify_batch for callers that cannot allocate device memory.
 *
 * The SDCP draft has no counterpart to this entry point: it exists for callers that must not
 * call cudaMalloc, such as code running inside a CUDA graph being built by someone else,
 * an allocator-less runtime, or a plugin whose host forbids device allocations.  Instead
 * of a caller-provided workspace it uses a scratch array of SDCP_NOALLOC_SCRATCH_BYTES that
 * lives in the library itself (a file-scope __device__ array): every GPU that loads the
 * library holds that memory until the process exits.  The caller still passes the inputs
 * and outputs, exactly as for sdcp_verify_batch, and gets identical results.
 *
 * Limit: sdcp_workspace_bytes(V, B, total_drafts) must not exceed
 * SDCP_NOALLOC_SCRATCH_BYTES; larger batches are rejected with SDCP_E_SCRATCH_LIMIT before
 * anything is launched.  The function calls no cudaMalloc, cudaFree or other allocating
 * routine.
 * Set-up: the first call on a device looks up the array's device address on the current
 * device (cudaGetSymbolAddress) and caches it; make that first call outside any stream
 * capture.  The current device must be the one the stream and the buffers belong to.
 * Sharing: all calls on a device share the one array and it keeps whatever the last call
 * left in it; nothing in it needs to start at zero.  Calls whose work overlaps on the GPU
 * (different streams, or host threads without ordering) race on the array: serialise them.
 * Returns as sdcp_verify_batch, plus SDCP_E_DEVICE if the device or the array's address
 * cannot be obtained.
 */
#define SDCP_NOALLOC_SCRATCH_BYTES ((size_t)2 << 20)
int sdcp_verify_batch_noalloc(const void* target_logits, const void* draft_logits, int dtype,
                              int64_t V, int32_t B, const int32_t* m_offsets,
                              int64_t total_drafts, const int32_t* draft_tokens,
                              const sdcp_session_params* params, int32_t* accepted,
                              int32_t* n_out, int32_t* out_tokens, int32_t* status,
                              void* stream);

/* ---- random values of the acceptance step --------------------------------------- */
#define SDCP_RNG_PHILOX4X32_10 0  /* counter-based Philox (the default, described above) */
#define SDCP_RNG_HMAC_SHA256   1  /* the draft's own derivation (Section 6.4, last
                                     paragraph): HMAC-SHA-256 keyed with the seed as eight
                                     octets in network order, over "SDCP-VERIFY-1" || 0x00
                                     || session (16 octets) || uint32(round) || uint32(i) ||
                                     uint8(purpose), the first 53 bits / 2^53; i is the
                                     1-based position of the pages (the acceptance test of
                                     0-based position k uses i = k + 1, the additional token
                                     after a accepted tokens i = a + 1) */

/* Options of sdcp_verify_batch_ex (host struct). */
typedef struct sdcp_verify_options {
  uint32_t struct_size;         /* sizeof(sdcp_verify_options) */
  uint32_t rng_id;              /* SDCP_RNG_* */
  const uint8_t* session_ids;   /* device, [B][16]: each session's 16-octet identifier
                                   (Section 5.2 session-id); needed by SDCP_RNG_HMAC_SHA256,
                                   ignored by Philox (which uses params[b].session_tag) */
  const float* q_rows;          /* device, [total_drafts][V] binary32, or NULL: q given as the
                                   drafter's rows of probabilities (Section 5.2 q_rows; q[i]
                                   is row i of the session, Section 6.4 Rule 2), used as given
                                   (no sampling profile).  Draft logits are then not read (they
                                   may be NULL) and the first phase reads target rows only.
                                   q(x) = 0 gives SDCP_S_BAD_PROPOSAL; a q(x) that is NaN,
                                   infinite or negative gives SDCP_S_BAD_PARAMS; other values
                                   of a row are used as given. */
} sdcp_verify_options;

/*
 * sdcp_verify_batch with options: the same arguments, layout and results, with the random
 * values chosen by opts->rng_id and q from the draft logits or from opts->q_rows.
 * opts = NULL is sdcp_verify_batch.  Returns SDCP_E_INVALID for an unknown rng_id, a
 * struct_size below sizeof(sdcp_verify_options), or the HMAC generator without session_ids;
 * SDCP_E_ALIGN for q_rows not aligned to 4 bytes.
 */
int sdcp_verify_batch_ex(const void* target_logits, const void* draft_logits, int dtype,
                         int64_t V, int32_t B, const int32_t* m_offsets, int64_t total_drafts,
                         const int32_t* draft_tokens, const sdcp_session_params* params,
                         int32_t* accepted, int32_t* n_out, int32_t* out_tokens,
                         int32_t* status, void* workspace, size_t workspace_bytes,
                         const sdcp_verify_options* opts, void* stream);

/* ---- the commit step after acceptance (Sections 4.2, 6.3, 6.5) ------------------- */
/* actions of a verdict (Section 4.1 "action"; Section 6.5.2) */
#define SDCP_ACTION_NONE        (-1) /* the session's status was not SDCP_S_OK: nothing
                                        committed, its state unchanged */
#define SDCP_ACTION_CONTINUE    0
#define SDCP_ACTION_REDUCE      1
#define SDCP_ACTION_SWITCH      2
#define SDCP_ACTION_SELF_DECODE 3
#define SDCP_ACTION_FINISH      4
#define SDCP_ACTION_FAIL        5
#define SDCP_NO_SELF_LOAD  0xFFFFFFFFu  /* the contract has no self_load member */

/* The contract terms of one session the commit step uses (Section 4.1), 48 bytes, device. */
typedef struct sdcp_commit_params {
  uint32_t max_new;       /* maximum output tokens of the session */
  uint32_t stop_offset;   /* its stop tokens are stop_tokens[stop_offset .. +stop_count) */
  uint32_t stop_count;
  uint32_t m_max;         /* upper bound on M (<= SDCP_MAX_M); caps m_cap */
  uint32_t low_rounds;    /* R >= 1, the escalation period */
  uint32_t low_ratio;     /* percent 0..100; 0 = absent (a round is low iff a = 0) */
  uint32_t self_load;     /* percent 0..100, or SDCP_NO_SELF_LOAD */
  uint32_t fallback_len;  /* 1..8 entries of fallback[] */
  uint8_t fallback[8];    /* the ladder: SDCP_ACTION_REDUCE, _SWITCH, _SELF_DECODE, _FAIL */
  uint32_t m_restore;     /* after a round that is not low, m_cap grows by this, up to m_max
                             (Section 6.5.1: "restore gradually"; 0 = never) */
  uint32_t reserved;
} sdcp_commit_params;

/* The verifier's per-session state between rounds, 64 bytes, device; read and updated. */
typedef struct sdcp_session_state {
  uint8_t digest[32];     /* d[n], the committed-prefix digest (Section 4.2) */
  uint32_t committed;     /* n, the committed length */
  uint32_t c, g, j;       /* consecutive low rounds, consecutive rounds not low, position in
                             the fallback list (Section 6.5.2) */
  uint32_t m_cap;         /* the largest M of the next round (Section 6.5.1); set it to
                             m_init before the first round */
  uint32_t reserved[3];
} sdcp_session_state;

/*
 * The commit step of one batch, after sdcp_verify_batch on the same stream (Section 6.3,
 * steps "Acceptance" (its truncation), "Commit" and "Control"; Sections 4.2 and 6.5).  For
 * each session b whose status is SDCP_S_OK:
 *   - truncation: the emitted tokens out_tokens[m_offsets[b] + b ..][0 .. n_out[b]) are
 *     cut after the first stop token of the session (the stop token itself is emitted)
 *     and to at most max_new - committed tokens; n_out[b] is lowered in place and the
 *     dropped slots set to -1;
 *   - commit: state.digest becomes d[n + m] by d[k] = SHA-256(d[k-1] || uint32(o[k])) over
 *     the m tokens kept, and state.committed grows by m;
 *   - control: the round is low if 100 a < low_ratio M (or, with low_ratio 0, if a = 0),
 *     with a = accepted[b] and M = m_offsets[b+1] - m_offsets[b]; the counters c, g, j and
 *     m_cap follow Section 6.5.2 (the ladder entry j applies when c reaches R, skipping
 *     self_decode unless self_load is present and load_percent <= self_load; "fail" when no
 *     entry remains; reduce halves m_cap, at least 1); a round that emitted a stop token or
 *     reached max_new gets SDCP_ACTION_FINISH instead (its counters are still updated, no
 *     ladder entry is applied).
 *   action[b] receives the SDCP_ACTION_* of the round (SDCP_ACTION_NONE for a session whose
 *   status is not SDCP_S_OK; its state, n_out and tokens are left as they are).
 * All pointers are device memory: m_offsets, accepted, status [B] / [B+1] as written by
 * sdcp_verify_batch; n_out, out_tokens in/out; cparams [B]; stop_tokens [sum of
 * stop_count] (may be NULL when every stop_count is 0); state [B] in/out; action [B] out.
 * Asynchronous on `stream`; allocates nothing.  Returns SDCP_OK, SDCP_E_INVALID (null
 * pointer, B < 0) or SDCP_E_LAUNCH.  Contract terms out of range (low_rounds 0,
 * fallback_len > 8) are read as the nearest valid value (1, 8).
 */
int sdcp_commit_batch(int32_t B, const int32_t* m_offsets, const int32_t* accepted,
                      int32_t* n_out, int32_t* out_tokens, const int32_t* status,
                      const sdcp_commit_params* cparams, const uint32_t* stop_tokens,
                      sdcp_session_state* state, uint32_t load_percent, int32_t* action,
                      void* stream);

/*
 * Host-side split of one ragged batch into n_parts contiguous blocks of sessions for
 * n_parts GPUs (one process per GPU).  Sessions are independent (Section 6.3 "Scoring":
 * a verifier may batch the proposals of many sessions), so block k can be verified on its
 * own GPU, and concatenating the blocks' outputs in order gives the whole batch's outputs:
 * no collective is needed on the data path.
 *
 * m_offsets  host, [B+1] int32 (as for sdcp_verify_batch).
 * params     host, [B] sdcp_session_params, or NULL (every session counted as Rule 2).
 * bounds     host out, [n_parts+1] int32: block k holds sessions bounds[k] .. bounds[k+1]-1;
 *            bounds[0] = 0, bounds[n_parts] = B, non-decreasing.
 * The blocks are balanced by the rows each session makes the first phase read: M_b + 1
 * target rows, plus M_b draft rows under Rule 2.  Boundary k is the first session index
 * (not before boundary k-1) whose prefix of rows comes closest to k/n_parts of the total;
 * the split is a pure function of its inputs.
 * Returns SDCP_OK, or SDCP_E_INVALID for null pointers, B < 0, n_parts < 1 or offsets that
 * are not non-decreasing from 0.  Touches no device.
 */
int sdcp_split_sessions(const int32_t* m_offsets, const sdcp_session_params* params, int32_t B,
                        int32_t n_parts, int32_t* bounds);

/* Human-readable text for an SDCP_E_* code (static storage, never NULL). */
const char* sdcp_strerror(int code);

/* ABI version of this header; bumps on any incompatible change. */
#define SDCP_ABI_VERSION 2
int sdcp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDCP_H */
