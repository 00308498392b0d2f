/*
 * clef_head.h — C ABI of the Clef JointSchemaHead forward pass on GB300 (sm_103a).
 *
 * The head turns the backbone's final-norm hidden states of a batch of encoded
 * records into one logit per option of every typed question, in one pass, then a
 * per-question softmax and the derived answers.  Sources (web pages, by title):
 *   "clef-4bit JointSchemaHead walkthrough" section 3 steps 1-4 (pooling, option
 *   query, evidence routing, field aggregation, joint layers, scorer);
 *   "Dissecting the Clef-Flash architecture" section 3.2 (head configuration);
 *   "clef-flash-CoreAI metadata.json" keys decision.spans, decision.option_order,
 *   decision.question_types, decision.head.reads, decision.head.lexical,
 *   decision.softmax, decision.response;
 *   "Clef-Flash inference tuning checklist" tip 1 (padding to the longest record)
 *   and tip 2 (schema budget errors).
 *
 * Conventions for every entry point:
 *   - Device pointers are caller-owned CUDA device memory; host pointers are
 *     caller-owned host memory, read during the call only.  The library never
 *     allocates or frees device memory: scratch lives in the caller's workspace.
 *   - bf16 tensors are passed as uint16_t bit patterns.  Matrices are row-major;
 *     weight matrices follow the torch Linear layout [out_features, in_features].
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  All work is enqueued asynchronously on it; outputs are valid once
 *     the stream reaches the call.
 *   - Every entry point returns a clef_status.  Arguments are validated on the
 *     host before anything is launched; on an error nothing is launched.
 *   - One call at a time per workspace: two calls that share a workspace and
 *     overlap on the GPU race on it.
 */
#ifndef CLEF_HEAD_H
#define CLEF_HEAD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CLEF_API __attribute__((visibility("default")))
#else
#define CLEF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum clef_status {
    CLEF_OK = 0,
    CLEF_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, bad span / type / option table */
    CLEF_ERR_WORKSPACE_TOO_SMALL = 2,
    CLEF_ERR_UNSUPPORTED_CONFIG = 3, /* shape outside what the kernels handle (see clef_config) */
    CLEF_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
    CLEF_ERR_DEVICE_BOUNDS = 5,      /* a kernel met an out-of-range index (a token id) and skipped it */
    CLEF_ERR_DEVICE_TIMEOUT = 6      /* a kernel's bounded wait ran out; it stopped and returned */
} clef_status;

/* Head hyper-parameters: the joint_head_config.json fields of "Dissecting the
 * Clef-Flash architecture" section 3.2 (hidden_size, width, heads, feedforward,
 * routing_layers, layers) plus the output-embedding vocabulary size.
 * Supported: hidden % 64 == 0 and 64 <= hidden <= 8192; width = 64 * heads and
 * width <= 2048; ffn % 64 == 0; 1 <= n_route <= 4; 0 <= n_joint <= 8; vocab >= 1.
 * Anything else -> CLEF_ERR_UNSUPPORTED_CONFIG. */
typedef struct clef_config {
    int32_t hidden;   /* H: backbone hidden size (4096, or 5120 for the wide backbone) */
    int32_t width;    /* D: head width (1024) */
    int32_t heads;    /* attention heads (16); head dim = width / heads must be 64 */
    int32_t ffn;      /* F: feedforward width (4096) */
    int32_t n_route;  /* EvidenceRoutingLayer count (2) */
    int32_t n_joint;  /* joint transformer layers (4) */
    int32_t vocab;    /* rows of the lexical (lm_head) table (248320) */
} clef_config;

/* The typed question schema of a padded batch, as the encoder records it
 * ("clef-flash-CoreAI metadata.json" decision.spans / option_order /
 * question_types).  All tables are HOST memory.
 *   lengths[b]      real rows of record b; rows 0..lengths[b]-1 are real, the rest
 *                   of the Lpad rows are right padding.  1 <= lengths[b] <= Lpad.
 *   q_rec[q]        record of question q; non-decreasing in q.
 *   q_type[q]       0 noul | 1 choice | 2 score.
 *   q_span[2q..]    instruction span [start, end) of question q, 0 <= start < end <= lengths[b].
 *   q_opt_off[q]    CSR offsets into the option table, q_opt_off[0] = 0,
 *                   q_opt_off[Q] = O; every question has >= 1 option, a noul
 *                   question exactly 2 (true, false), at most 256 per question.
 *   o_span[2j..]    option span [start, end) of option j, same bounds as q_span.
 * Every record must own at least one question and at most 48 (more ->
 * CLEF_ERR_UNSUPPORTED_CONFIG).  Invalid tables -> CLEF_ERR_INVALID_ARGUMENT. */
typedef struct clef_schema {
    int32_t B;                 /* records */
    int32_t Lpad;              /* padded rows per record */
    int64_t row_stride;        /* elements between consecutive hidden rows: >= hidden, % 8 == 0 */
    const int32_t* lengths;    /* [B] */
    int32_t Q;                 /* questions */
    const int32_t* q_rec;      /* [Q] */
    const int32_t* q_type;     /* [Q] */
    const int32_t* q_span;     /* [Q][2] */
    const int32_t* q_opt_off;  /* [Q+1] */
    int32_t O;                 /* options */
    const int32_t* o_span;     /* [O][2] */
} clef_schema;

/* Number of tensors in the weight pointer table for `cfg`
 * (6 + 16 * n_route + 9 + 12 * n_joint + 8), or -1 for an unsupported config.
 * The table holds device bf16 tensors in this order (torch Linear layout):
 *   mem_ln.weight [H], mem_ln.bias [H],
 *   query.ctx.weight [D,H], query.lex.weight [D,H], query.question.weight [D,H], query.bias [D],
 *   per routing layer l:  attn_ln.weight [D], attn_ln.bias [D], q.weight [D,D], q.bias [D],
 *       k.weight [D,H], k.bias [D], v.weight [D,H], v.bias [D], o.weight [D,D], o.bias [D],
 *       ffn_ln.weight [D], ffn_ln.bias [D], ffn1.weight [F,D], ffn1.bias [F],
 *       ffn2.weight [D,F], ffn2.bias [D],
 *   option_ln.weight [D], option_ln.bias [D], field.pool.weight [1,D], field.pool.bias [1],
 *   field.question.weight [D,H], field.summary.weight [D,D], field.global.weight [D,H],
 *   field.bias [D], field.type_embedding [3,D],
 *   per joint layer i:  attn_ln.weight [D], attn_ln.bias [D], qkv.weight [3D,D], qkv.bias [3D],
 *       o.weight [D,D], o.bias [D], ffn_ln.weight [D], ffn_ln.bias [D],
 *       ffn1.weight [F,D], ffn1.bias [F], ffn2.weight [D,F], ffn2.bias [D],
 *   field_ln.weight [D], field_ln.bias [D], scorer.gate [1], scorer.joint_scale [1],
 *   scorer.mlp1.weight [D,4D], scorer.mlp1.bias [D], scorer.mlp2.weight [1,D], scorer.mlp2.bias [1].
 * Every pointer must be 16-byte aligned. */
CLEF_API int clef_weight_count(const clef_config* cfg);

/* Bytes of the derived-weight buffer that clef_prepare_weights fills. */
CLEF_API int clef_prepared_size(const clef_config* cfg, size_t* bytes);

/* Builds derived weights on the GPU (no host arithmetic):
 *   - memory K/V projections of every routing layer with the memory LayerNorm folded
 *     in: W' = W diag(gamma) (bf16), c = row sums of W' and b' = W beta + b (fp32),
 *     so that K = rstd (h W'^T - mu c) + b' equals W LN(h) + b;
 *   - the three option-query projections side by side [D, 3H];
 *   - the three field projections side by side [D, 2H + D].
 * `weights` is a host array of clef_weight_count(cfg) device pointers.
 * `prepared` is caller-owned device memory of clef_prepared_size bytes, 256-byte aligned. */
CLEF_API int clef_prepare_weights(const clef_config* cfg, const void* const* weights,
                         void* prepared, size_t prepared_bytes, void* stream);

/* Workspace bytes clef_head_forward needs for this schema. */
CLEF_API int clef_workspace_size(const clef_config* cfg, const clef_schema* schema, size_t* bytes);

/* Optional intermediate outputs (device pointers, NULL = not written), for
 * diagnosis and stage-wise parity checks. */
typedef struct clef_debug_outputs {
    float* pooled_u;      /* [Q][H] question vectors u_q */
    float* pooled_c;      /* [O][H] option context vectors c_j */
    float* pooled_x;      /* [O][H] option lexical vectors x_j */
    float* global_g;      /* [B][H] global vectors g_b */
    float* option_final;  /* [O][D] option vectors after routing and the final option LayerNorm */
    float* field_final;   /* [Q][D] field vectors after the joint layers and the final field LayerNorm */
    /* Optional cudaEvent_t handles (NULL = not recorded), recorded on `stream`
     * immediately before / after one kernel: [0] [1] the memory K/V projection GEMM,
     * [2] [3] the first routing layer's split-L attention kernel, [4] [5] span
     * pooling; [6] [7] are not recorded (the memory row statistics are computed by
     * the K/V projection, which [0] [1] bracket). */
    void* events[8];
    /* Optional launch timeline: when `timeline` is not NULL, the call records
     * timeline[k] (a cudaEvent_t) on `stream` right after its k-th kernel launch,
     * for k < timeline_len; the number of launches is written to *timeline_count. */
    void** timeline;
    int32_t timeline_len;
    int32_t* timeline_count;
    /* Which kernels run the per-record tail (option LayerNorm to softmax): 0 or 1, the
     * batched chain (one GEMM per projection over the whole batch, the faster one on
     * GB300); 2, one fused launch of a 16-CTA thread-block cluster per record group,
     * where the head shape allows it (width 1024, 16 heads, FFN 4096, at most 256
     * options per record).  The outputs agree within the parity tolerance either way. */
    int32_t tail_mode;
    /* Optional fp32 [R] each (NULL = not written): the memory LayerNorm statistics of
     * every compact row as the K/V projection computed them (mean, 1/sqrt(var + 1e-5)).
     * Record b's row t < lengths[b] is compact row R_b + t, R_b = the sum over b' < b of
     * lengths[b'] rounded up to a multiple of 128, and R = that sum over every record;
     * the round-up rows hold 0. */
    float* row_mu;
    float* row_rstd;
} clef_debug_outputs;

/* The forward pass.
 *   hidden     device bf16 [B, Lpad, H] with row stride schema->row_stride elements
 *              (record stride Lpad * row_stride): the backbone's final-norm hidden
 *              states ("clef-flash-CoreAI metadata.json" decision.head.reads).
 *              16-byte aligned.
 *   token_ids  device int32 [B, Lpad]: the prompt's token ids; the lexical vector of
 *              an option reads the ids under its span.  An id outside [0, vocab) is
 *              skipped and reported as CLEF_ERR_DEVICE_BOUNDS by clef_device_status.
 *   lexical    device bf16 [vocab, H]: the untied output-embedding table.
 *   weights    host array of device pointers (see clef_weight_count).
 *   prepared   device buffer filled by clef_prepare_weights for the same weights.
 *   logits, probs  device fp32 [O]: per-option logit and per-question softmax probability.
 *   q_value    device fp32 [Q]: noul p(true); choice max p; score sum(level * p).
 *   q_conf     device fp32 [Q]: max p of the question.
 *   q_argmax   device int32 [Q]: index of the first maximum within the question's options.
 *   workspace  device scratch of clef_workspace_size bytes, 256-byte aligned.
 *   debug      optional (NULL) intermediate outputs.
 * Host-side validation errors return before any launch.  The call does not wait
 * for the GPU: device-side bound / timeout flags are read by clef_device_status.
 * Every device step of a call without `debug` is a kernel launch on `stream`, so
 * after one ordinary call with the same arguments the call can be captured into a
 * CUDA graph; each replay uploads the captured plan, clears the status word and the
 * memory statistics' flags, and recomputes the whole head from the buffers' contents
 * at replay time. */
CLEF_API int clef_head_forward(const clef_config* cfg, const void* const* weights, const void* prepared,
                      const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                      const uint16_t* lexical, float* logits, float* probs, float* q_value,
                      float* q_conf, int32_t* q_argmax, void* workspace, size_t workspace_bytes,
                      const clef_debug_outputs* debug, void* stream);

/* Streaming memory ingestion.  A backbone may produce the final-norm hidden rows of a
 * record in chunks ("clef-flash-CoreAI metadata.json" decision.readout: a row of T ids
 * runs as ceil(T / 64) calls of 64 positions, whose hidden rows are concatenated).  The
 * schema (and so every record's final length and spans) is known before the first
 * chunk, because the encoder lays the whole prompt out first.  The memory part of the
 * head (row statistics and the K/V projection, its dominant cost) can then run chunk
 * by chunk while the backbone produces later rows:
 *   clef_stream_begin   once per batch: validates the schema, uploads its launch plan
 *                       into `workspace` and clears the status word;
 *   clef_stream_rows    whenever rows [row0, row0 + n_rows) of record `record` are
 *                       final in `hidden` (same layout as for clef_head_forward):
 *                       computes their statistics and K/V into the workspace.  Chunks
 *                       of any size, in any order; every real row exactly once.
 *                       0 <= row0, 1 <= n_rows, row0 + n_rows <= lengths[record].
 *   clef_stream_finish  after every real row of every record went through
 *                       clef_stream_rows: the rest of the head (pooling, routing,
 *                       fields, joint layers, scorer, softmax), with the same arguments
 *                       and outputs as clef_head_forward.
 * The outputs equal clef_head_forward's on the same inputs.  All calls of one batch use
 * the same schema, prepared weights and workspace (sized by clef_workspace_size), on
 * one stream; the workspace must not be used by other calls in between. */
CLEF_API int clef_stream_begin(const clef_config* cfg, const clef_schema* schema, void* workspace,
                               size_t workspace_bytes, void* stream);
CLEF_API int clef_stream_rows(const clef_config* cfg, const void* prepared, const clef_schema* schema,
                              const uint16_t* hidden, int32_t record, int32_t row0, int32_t n_rows,
                              void* workspace, size_t workspace_bytes, void* stream);
CLEF_API int clef_stream_finish(const clef_config* cfg, const void* const* weights, const void* prepared,
                                const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                                const uint16_t* lexical, float* logits, float* probs, float* q_value,
                                float* q_conf, int32_t* q_argmax, void* workspace, size_t workspace_bytes,
                                const clef_debug_outputs* debug, void* stream);

/* Streaming ingestion of fp16 hidden rows ("clef-flash-CoreAI metadata.json"
 * decision.readout: the chunked graph hands over 64-position chunks of fp16 hidden
 * rows).  Same arguments, layout and rules as clef_stream_rows / clef_stream_finish,
 * but `hidden` holds IEEE fp16 values instead of bf16.  Every fp16 value is rounded to
 * bf16 (round to nearest even) where the head reads it -- the memory statistics, the
 * K/V projection and the span pooling -- so the outputs equal those of the bf16 calls
 * on the rounded rows, bit for bit.  clef_stream_rows_f16 rounds a chunk through a
 * staging area inside the workspace, at most 1024 rows per pass; it needs no extra
 * workspace beyond clef_workspace_size.  The two entry points pair with each other:
 * a batch whose rows came in as fp16 is finished with clef_stream_finish_f16, which
 * reads `hidden` (fp16) again for the pooled spans and the global row. */
CLEF_API int clef_stream_rows_f16(const clef_config* cfg, const void* prepared, const clef_schema* schema,
                                  const uint16_t* hidden, int32_t record, int32_t row0, int32_t n_rows,
                                  void* workspace, size_t workspace_bytes, void* stream);
CLEF_API int clef_stream_finish_f16(const clef_config* cfg, const void* const* weights, const void* prepared,
                                    const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                                    const uint16_t* lexical, float* logits, float* probs, float* q_value,
                                    float* q_conf, int32_t* q_argmax, void* workspace, size_t workspace_bytes,
                                    const clef_debug_outputs* debug, void* stream);

/* Waits for `stream`, then reads and clears the device-side status word kept at the
 * start of `workspace`: CLEF_OK, CLEF_ERR_DEVICE_BOUNDS or CLEF_ERR_DEVICE_TIMEOUT.
 * Every clef_head_forward / clef_span_sums call clears that word when it starts, so
 * the status covers the latest call on the workspace. */
CLEF_API int clef_device_status(void* workspace, void* stream);

/* Self-test of the device-side wait limits (the pages have no counterpart: this is a
 * property of this implementation).  Clears the first 256 bytes of `workspace` (device
 * memory, 256-byte aligned, at least 256 bytes) and launches one kernel whose single
 * waiting thread waits, for `limit_ns` nanoseconds (1 us .. 100 ms) each, first on a
 * shared-memory barrier that never completes, then on a global flag (at byte 128 of
 * the workspace) that nothing sets.  Each wait gives up, sets the timeout bit and
 * records itself in the int32 at byte 8 of the workspace (bit 0: the barrier wait,
 * bit 1: the flag wait); the kernel returns.  clef_device_status then reports
 * CLEF_ERR_DEVICE_TIMEOUT and the CUDA context stays usable.  Every wait of the head's
 * own kernels has one of these two forms, with a 2 s limit.
 * Returns CLEF_ERR_INVALID_ARGUMENT for a null or misaligned workspace or a limit out
 * of range, CLEF_ERR_CUDA if the launch fails, else CLEF_OK (asynchronously). */
CLEF_API int clef_selftest_wait_timeout(void* workspace, int64_t limit_ns, void* stream);

/* Index check of the pooling step ("clef-4bit JointSchemaHead walkthrough" section 3
 * step 1): un-normalised fp32 sums of the raw hidden rows over every instruction span
 * (q_sum [Q][H]) and option span (o_sum [O][H]) and of the lexical rows under every
 * option span (x_sum [O][H]), each summed in row order.  With small-integer inputs
 * the sums are exact, so they check span, offset and gather indexing bit for bit.
 * `workspace` as for clef_head_forward. */
CLEF_API int clef_span_sums(const clef_config* cfg, const clef_schema* schema, const uint16_t* hidden,
                   const int32_t* token_ids, const uint16_t* lexical, float* q_sum, float* o_sum,
                   float* x_sum, void* workspace, size_t workspace_bytes, void* stream);

/* Largest scratch the allocation-free span-sum entry point below can use. */
#define CLEF_SPAN_SUMS_NOALLOC_SCRATCH_BYTES (1u << 20)

/* clef_span_sums for callers that cannot allocate device memory.  The pages have
 * no counterpart of this entry point; it exists for callers that must not call
 * cudaMalloc themselves: code that runs inside another runtime's fixed device-memory
 * pool, a plug-in that is handed only its input and output buffers, or code paths
 * where a device allocation would stall or fail.  Such callers cannot provide the
 * workspace clef_span_sums needs.
 *   - The scratch (the launch plan of the batch and the device status word) lives in
 *     one static device array of CLEF_SPAN_SUMS_NOALLOC_SCRATCH_BYTES (1 MiB) inside
 *     the library.  Every GPU that loads the library holds that array until the
 *     process exits.  A schema whose plan does not fit returns
 *     CLEF_ERR_WORKSPACE_TOO_SMALL before anything is launched.  The plan takes 36
 *     bytes per question, 32 per option, 40 per record, 8 per 128 memory rows and 16
 *     per 1024 memory rows (more for records with over 64 options), so 1 MiB holds,
 *     for example, 1 500 questions and 15 000 options over 256 records of 16 384
 *     rows.
 *   - The caller passes inputs and outputs exactly as for clef_span_sums, and gets
 *     the same sums bit for bit.
 *   - Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *   - The plan reaches the array as kernel parameters of small upload kernels, so no
 *     host buffer is pinned or kept.
 *   - The first call on a device looks up the device address of the array with
 *     cudaGetSymbolAddress, with that device current.  Make that first call before
 *     any stream capture.
 *   - The call waits for `stream` before it returns, so that it can return a
 *     device-side index error (CLEF_ERR_DEVICE_BOUNDS) directly.
 *   - Every call uses the same array.  The status word is cleared at the start of
 *     each call and the plan is rewritten, so nothing of an earlier call leaks into
 *     a later one; but two calls that overlap on the GPU (other host threads, other
 *     streams) race on the array and must be serialised by the caller. */
CLEF_API int clef_span_sums_noalloc(const clef_config* cfg, const clef_schema* schema, const uint16_t* hidden,
                                    const int32_t* token_ids, const uint16_t* lexical, float* q_sum,
                                    float* o_sum, float* x_sum, void* stream);

/* The dense-contraction kernel of the head on its own (tcgen05 / TMEM, TMA-fed):
 *   C[m][n] = sum_k A[m][k] * B[n][k] (+ bias[n]),  fp32 out, m < M, n < N.
 * A bf16 [M][K] row stride lda, B bf16 [N][K] row stride ldb, bias fp32 [N] or NULL,
 * C fp32 row stride ldc.  K % 64 == 0, lda % 8 == 0, ldb % 8 == 0, N % 64 == 0,
 * A and B 16-byte aligned.  `flags` is a device int32 that receives the
 * CLEF_ERR_DEVICE_TIMEOUT bit (1 << 1) if a bounded wait runs out. */
CLEF_API int clef_gemm_bf16(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                   const float* bias, float* C, int64_t ldc, int32_t M, int32_t N, int32_t K,
                   int32_t* flags, void* stream);

/* Number of kernels this library has launched in this process so far. */
CLEF_API uint64_t clef_kernel_launches(void);

/* Human-readable name of a status code. */
CLEF_API const char* clef_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CLEF_HEAD_H */
