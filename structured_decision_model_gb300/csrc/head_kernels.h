// Argument blocks and launchers of the head's non-GEMM kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace clef {

constexpr int kAttnChunk = 1024;  // memory rows per split-L routing-attention work item
constexpr int kAttnQRows = 64;    // option queries per routing-attention work item
constexpr int kMaxFields = 48;    // questions per record handled by the field self-attention kernel
constexpr int kMaxOptions = 256;  // options per question
constexpr int kPlanChunkInts = 8000;  // plan ints carried by one upload launch (32 KB of parameters)

struct SpanPoolArgs {
    const uint16_t* hidden; int64_t row_stride; int Lpad; int H; int vocab;
    const int32_t* token_ids; const uint16_t* lexical;
    const float* mu; const float* rstd;          // compact-row statistics
    const uint16_t* ln_w; const uint16_t* ln_b;  // memory LayerNorm affine
    const int4* items;                           // per item {kind << 30 | index, record, span start, span end}
    const int32_t* lengths; const int32_t* rec_row_off; const int32_t* rec_q_off;
    const int32_t* q_rec; const int32_t* q_span; const int32_t* q_opt_off;
    const int32_t* o_rec; const int32_t* o_span;
    // pooled outputs
    uint16_t* a_query; int64_t ld_query;  // [O][3H]: c | x | u_q(j)
    uint16_t* a_field; int64_t ld_field;  // [Q][2H + D]: u | g | summary
    float* u32; float* x32; float* g32;   // fp32 copies for the scorer
    float* dbg_c;                         // optional [O][H]
    // raw-sum mode
    float* q_sum; float* o_sum; float* x_sum;
    int* flags;
    int in_f16;                           // hidden rows are fp16 (rounded to bf16 when read)
};

struct RouteAttnArgs {
    const uint16_t* q; int64_t ldq;       // [O][D] bf16 queries
    const uint16_t* kv; int64_t ldkv;     // [R][ldkv] bf16 memory keys / values
    int64_t kv_rows;                      // R
    int k_col, v_col;                     // column of this layer's K and V blocks
    int heads;
    float scale_log2;                     // log2(e) / sqrt(head dim)
    const int32_t* chunk_rec; const int32_t* chunk_idx;  // per chunk: record, chunk index in the record
    const int32_t* unit_cx; const int32_t* unit_qp;      // per work unit: chunk, block of kAttnQRows options
    int n_units;
    const int32_t* lengths; const int32_t* rec_row_off; const int32_t* rec_o_off;
    const int64_t* rec_part_off;
    const int32_t* o_rec;
    float* pm; float* pl; float* pacc;    // partials
    uint16_t* out; int64_t ldo;           // [O][D] bf16 merged output
    int* flags;                           // device status word
};

struct ScoreArgs {
    int H, D;
    const int32_t* q_rec; const int32_t* q_type; const int32_t* q_opt_off;
    const float* u32; const float* g32; const float* x32;
    const float* f_hat; const float* o_hat;
    const uint16_t* mlp_hidden;           // [O][D] bf16, GELU(W1 z + b1)
    const uint16_t* w2; const uint16_t* b2; const uint16_t* gate; const uint16_t* joint_scale;
    float* logits; float* probs; float* q_value; float* q_conf; int32_t* q_argmax;
};

struct FoldArgs {
    int H, D;
    const uint16_t* w[8];                 // K / V weights of every routing layer, [D][H]
    const uint16_t* bias[8];
    const uint16_t* gamma; const uint16_t* beta;
    uint16_t* out_w; float* out_c; float* out_b;
};

// The per-record tail of the head (option LayerNorm, field aggregation, the joint
// layers, the field LayerNorm and the scorer with the softmax), one thread-block
// cluster per record.  Weights are bf16; the joint layers' pointers are per layer.
constexpr int kTailMaxJoint = 8;
constexpr int kTailMaxRecOptions = 256;  // options of one record the fused tail holds at once

struct RecordTailArgs {
    int B, H, D, F, n_joint, Q, O;
    int n_groups; const int32_t* grp_rec;   // cluster g runs records [grp_rec[g], grp_rec[g + 1])
    int* flags;                             // device status word (bounded-wait timeouts)
    const int32_t* rec_q_off; const int32_t* rec_o_off; const int32_t* q_type; const int32_t* q_rec;
    const int32_t* q_opt_off; const int32_t* o_q;
    // inputs
    const float* o_res;                     // [O][D] option stream after routing
    const float* u32; const float* g32; const float* x32;  // pooled vectors (fp32)
    uint16_t* a_field; int64_t ld_field;    // [Q][2H + D] bf16: u | g (read) | summary (written)
    // weights
    // weights: projection matrices in the sliced layout of launch_tail_slices (each
    // cluster CTA's rows as contiguous pre-swizzled 64-column tiles), vectors as given
    const uint16_t* opt_ln_w; const uint16_t* opt_ln_b;
    const uint16_t* pool_w; const uint16_t* pool_b;
    const uint16_t* w_field; const uint16_t* b_field; const uint16_t* type_emb;  // sliced [D][2H + D], [D], [3][D]
    const uint16_t* ln1_w[kTailMaxJoint]; const uint16_t* ln1_b[kTailMaxJoint];
    const uint16_t* w_qkv[kTailMaxJoint]; const uint16_t* b_qkv[kTailMaxJoint];  // sliced [3D][D]
    const uint16_t* w_o[kTailMaxJoint]; const uint16_t* b_o[kTailMaxJoint];      // sliced [D][D]
    const uint16_t* ln2_w[kTailMaxJoint]; const uint16_t* ln2_b[kTailMaxJoint];
    const uint16_t* w_1[kTailMaxJoint]; const uint16_t* b_1[kTailMaxJoint];      // sliced [F][D]
    const uint16_t* w_2[kTailMaxJoint]; const uint16_t* b_2[kTailMaxJoint];      // sliced [D][F]
    const uint16_t* fld_ln_w; const uint16_t* fld_ln_b;
    const uint16_t* gate; const uint16_t* joint_scale;
    const uint16_t* mlp1_w; const uint16_t* mlp1_b; const uint16_t* mlp2_w; const uint16_t* mlp2_b;  // mlp1 sliced [D][4D]
    // scratch (workspace) and outputs
    float* o_hat;                           // [O][D] fp32 (written)
    float* f_hat;                           // [Q][D] fp32 (written)
    uint16_t* ln_buf;                       // [Q][D] bf16
    uint16_t* attn_buf;                     // [Q][D] bf16
    uint16_t* hid_buf;                      // [Q][F] bf16
    uint16_t* z;                            // [O][4D] bf16
    float* logits; float* probs; float* q_value; float* q_conf; int32_t* q_argmax;
};

// Clusters of the fused tail the GPU holds at once (0: the fused tail is unavailable).
int record_tail_clusters();
// Whether the fused tail is built for this head shape (width 1024, 16 heads, FFN 4096).
bool record_tail_shape(int H, int D, int heads, int F, int n_joint);
cudaError_t launch_record_tail(const RecordTailArgs& a, cudaStream_t s);
// The sliced weight layout of the fused tail: W [N][K] (row stride K) becomes, for each
// of the 16 cluster CTAs r and each 64-column chunk kc, a tile of R rows x 128 bytes
// (1024-byte aligned, 16-byte chunks in the 128-byte swizzle), tiles of one CTA
// consecutive.  Row j of CTA r's tiles is W row r R + j (qkv = 0), or, for the fused
// q / k / v matrix (qkv = 1, R = 3 * 64), row (j / 64) D + 64 r + j % 64.
cudaError_t launch_tail_slices(const uint16_t* w, int K, int R, int qkv, int D, uint16_t* dst, cudaStream_t s);

cudaError_t launch_wait_timeout_selftest(int* flags, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_zero_slack(uint16_t* kv, int ldkv, const int32_t* rec_row_off, const int32_t* lengths, int B,
                              cudaStream_t s);
cudaError_t launch_span_pool(const SpanPoolArgs& a, int n_items, bool raw, cudaStream_t s);
cudaError_t launch_f16_rows_to_bf16(const uint16_t* src, int64_t ld_src, int rows, int H, uint16_t* dst,
                                    cudaStream_t s);
// A residual-stream projection finished from its deferred split-K partial products,
// followed by a LayerNorm: x = sum_s part[s] + bias + row_table[row_idx] (+ x when
// resid), the stream x updated, then LN(x) with (ln_w, ln_b) into out_bf16 / out_f32.
struct LnAccArgs {
    float* x = nullptr;                   // [rows][D] fp32 stream (read when resid, always written)
    int rows = 0, D = 0;
    const float* part = nullptr;          // S slabs [rows][D], slab stride part_stride elements
    int64_t part_stride = 0;
    int S = 0;
    const uint16_t* bias = nullptr;       // [D] bf16 or null
    const uint16_t* row_table = nullptr;  // [*][ld_table] bf16 rows added by row_idx[r], or null
    const int32_t* row_idx = nullptr;
    int64_t ld_table = 0;
    int resid = 0;
    const uint16_t* ln_w = nullptr;
    const uint16_t* ln_b = nullptr;
    uint16_t* out_bf16 = nullptr;         // [rows][D] or null
    float* out_f32 = nullptr;             // [rows][D] or null
    // scorer MLP input rows z_j = [y_q, o_hat_j, y_q * o_hat_j, |y_q - o_hat_j|] (bf16
    // [O][4D]) for the options j of row q (z_opt_off[q] .. z_opt_off[q + 1]), or null
    uint16_t* z = nullptr;
    const int32_t* z_opt_off = nullptr;
    const float* z_o_hat = nullptr;       // [O][D]
};
cudaError_t launch_layer_norm_acc(const LnAccArgs& a, cudaStream_t s);
cudaError_t launch_route_attn_partial(const RouteAttnArgs& a, int O,
                                      cudaStream_t s);
cudaError_t launch_route_attn_merge(const RouteAttnArgs& a, int O, cudaStream_t s);
cudaError_t launch_field_pool(const float* o_hat, int D, const int32_t* q_opt_off, int Q, const uint16_t* w_a,
                              const uint16_t* b_a, uint16_t* out, int64_t ldo, int col_off, cudaStream_t s);
cudaError_t launch_field_attn(const uint16_t* qkv, int D, int heads, const int32_t* rec_q_off, int B, float scale,
                              uint16_t* out, cudaStream_t s);
cudaError_t launch_score_softmax(const ScoreArgs& a, int Q, cudaStream_t s);
cudaError_t launch_fold_kv(const FoldArgs& a, int rows, cudaStream_t s);
// Copies the plan (n int32 values) to dst and clears z0 / z1 (16-byte aligned, sizes
// multiples of 16 bytes; null with size 0 when unused).
cudaError_t launch_plan_upload(int32_t* dst, const int32_t* src, size_t n, void* z0, size_t z0_bytes, void* z1,
                               size_t z1_bytes, cudaStream_t s);
cudaError_t launch_copy_cols(uint16_t* dst, int64_t ld_dst, int col_off, const uint16_t* src, int64_t ld_src,
                             int rows, int cols, cudaStream_t s);

}  // namespace clef
