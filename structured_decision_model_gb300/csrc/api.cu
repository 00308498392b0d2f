// C ABI of the Clef JointSchemaHead forward pass: host-side validation, the
// launch plan of one batch, the workspace layout and the launch sequence.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/clef_head.h"
#include "common.cuh"
#include "head_kernels.h"
#include "kernels.h"

using namespace clef;

namespace {

constexpr int kTile = 128;  // rows per GEMM output tile; records are padded to it in compact row space
constexpr int kStageRows = 1024;  // fp16 streaming: rows rounded to bf16 per staging pass

bool config_ok(const clef_config* c) {
    if (!c) return false;
    if (c->hidden < 64 || c->hidden > 8192 || c->hidden % 64) return false;
    if (c->heads < 1 || c->width != 64 * c->heads || c->width > 2048) return false;
    if (c->ffn < 64 || c->ffn % 64) return false;
    if (c->n_route < 1 || c->n_route > 4 || c->n_joint < 0 || c->n_joint > 8) return false;
    if (c->vocab < 1) return false;
    return true;
}

struct WIdx {
    int nr, nj;
    explicit WIdx(const clef_config* c) : nr(c->n_route), nj(c->n_joint) {}
    int route(int l, int k) const { return 6 + 16 * l + k; }
    int mid(int k) const { return 6 + 16 * nr + k; }
    int joint(int i, int k) const { return 6 + 16 * nr + 9 + 12 * i + k; }
    int tail(int k) const { return 6 + 16 * nr + 9 + 12 * nj + k; }
    int count() const { return 6 + 16 * nr + 9 + 12 * nj + 8; }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Carve {
    size_t off = 0;
    size_t take(size_t bytes) {
        size_t o = off;
        off = align256(off + bytes);
        return o;
    }
};

struct PreparedLayout {
    size_t wkv, ckv, bkv, wq0, wfield, total;
    // the fused tail's sliced copies (launch_tail_slices), for the head shapes it supports
    bool tail = false;
    size_t t_field = 0, t_mlp1 = 0, t_qkv[kTailMaxJoint] = {}, t_o[kTailMaxJoint] = {}, t_w1[kTailMaxJoint] = {},
           t_w2[kTailMaxJoint] = {};
    PreparedLayout(const clef_config* c) {
        const size_t H = c->hidden, D = c->width, F = c->ffn, NKV = size_t(2) * c->n_route * D;
        Carve cv;
        wkv = cv.take(NKV * H * 2);
        ckv = cv.take(NKV * 4);
        bkv = cv.take(NKV * 4);
        wq0 = cv.take(D * 3 * H * 2);
        wfield = cv.take(D * (2 * H + D) * 2);
        tail = record_tail_shape(c->hidden, c->width, c->heads, c->ffn, c->n_joint);
        if (tail) {
            t_field = cv.take(D * (2 * H + D) * 2);
            t_mlp1 = cv.take(D * 4 * D * 2);
            for (int i = 0; i < c->n_joint; ++i) {
                t_qkv[i] = cv.take(3 * D * D * 2);
                t_o[i] = cv.take(D * D * 2);
                t_w1[i] = cv.take(F * D * 2);
                t_w2[i] = cv.take(D * F * 2);
            }
        }
        total = cv.off;
    }
};

// Host-built plan of one batch: tables the kernels index, and sizes.
struct Plan {
    int B = 0, Q = 0, O = 0, R = 0, n_mtiles = 0, n_items = 0, n_chunks = 0, n_units = 0, max_rec_options = 0;
    int n_groups = 0;  // record groups of the fused tail (plan_tail_groups)
    int64_t P = 0;  // attention partial rows
    std::vector<int32_t> blob;  // int32 tables followed by the int64 partial offsets
    // offsets (in int32 units) of each table in the blob
    size_t lengths, rec_row_off, rec_q_off, rec_o_off, q_rec, q_type, q_span, q_opt_off, o_rec, o_q, o_span,
        tile_rec, tile_a_row, item, chunk_rec, chunk_idx, unit_cx, unit_qp, rec_part_off, grp_rec;
};

int validate_schema(const clef_config* c, const clef_schema* s) {
    if (!s || !s->lengths || !s->q_rec || !s->q_type || !s->q_span || !s->q_opt_off || !s->o_span)
        return CLEF_ERR_INVALID_ARGUMENT;
    if (s->B < 1 || s->Lpad < 1 || s->Q < 1 || s->O < 1) return CLEF_ERR_INVALID_ARGUMENT;
    if (s->row_stride < c->hidden || s->row_stride % 8) return CLEF_ERR_INVALID_ARGUMENT;
    if (int64_t(s->B) * s->Lpad >= (int64_t(1) << 31)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    for (int b = 0; b < s->B; ++b)
        if (s->lengths[b] < 1 || s->lengths[b] > s->Lpad) return CLEF_ERR_INVALID_ARGUMENT;
    if (s->q_opt_off[0] != 0 || s->q_opt_off[s->Q] != s->O) return CLEF_ERR_INVALID_ARGUMENT;
    std::vector<int> per_rec(s->B, 0);
    for (int q = 0; q < s->Q; ++q) {
        const int b = s->q_rec[q];
        if (b < 0 || b >= s->B) return CLEF_ERR_INVALID_ARGUMENT;
        if (q > 0 && b < s->q_rec[q - 1]) return CLEF_ERR_INVALID_ARGUMENT;
        ++per_rec[b];
        const int t = s->q_type[q];
        if (t < 0 || t > 2) return CLEF_ERR_INVALID_ARGUMENT;
        const int st = s->q_span[2 * q], en = s->q_span[2 * q + 1];
        if (st < 0 || st >= en || en > s->lengths[b]) return CLEF_ERR_INVALID_ARGUMENT;
        const int n = s->q_opt_off[q + 1] - s->q_opt_off[q];
        if (n < 1 || n > kMaxOptions) return CLEF_ERR_INVALID_ARGUMENT;
        if (t == 0 && n != 2) return CLEF_ERR_INVALID_ARGUMENT;
        for (int j = s->q_opt_off[q]; j < s->q_opt_off[q + 1]; ++j) {
            const int os = s->o_span[2 * j], oe = s->o_span[2 * j + 1];
            if (os < 0 || os >= oe || oe > s->lengths[b]) return CLEF_ERR_INVALID_ARGUMENT;
        }
    }
    for (int b = 0; b < s->B; ++b) {
        if (per_rec[b] < 1) return CLEF_ERR_INVALID_ARGUMENT;
        if (per_rec[b] > kMaxFields) return CLEF_ERR_UNSUPPORTED_CONFIG;
    }
    return CLEF_OK;
}

void build_plan(const clef_config* c, const clef_schema* s, Plan& p) {
    p.B = s->B;
    p.Q = s->Q;
    p.O = s->O;
    std::vector<int32_t>& v = p.blob;
    v.clear();
    auto put = [&](size_t n) {
        size_t o = v.size();
        v.resize(o + n, 0);
        return o;
    };
    const int B = s->B, Q = s->Q, O = s->O;
    p.lengths = put(B);
    p.rec_row_off = put(B + 1);
    p.rec_q_off = put(B + 1);
    p.rec_o_off = put(B + 1);
    p.q_rec = put(Q);
    p.q_type = put(Q);
    p.q_span = put(2 * size_t(Q));
    p.q_opt_off = put(Q + 1);
    p.o_rec = put(O);
    p.o_q = put(O);
    p.o_span = put(2 * size_t(O));
    int R = 0;
    int nch = 0;
    for (int b = 0; b < B; ++b) {
        v[p.lengths + b] = s->lengths[b];
        v[p.rec_row_off + b] = R;
        R += (s->lengths[b] + kTile - 1) / kTile * kTile;
        nch += (s->lengths[b] + kAttnChunk - 1) / kAttnChunk;
    }
    v[p.rec_row_off + B] = R;
    p.R = R;
    p.n_mtiles = R / kTile;
    std::vector<int> rq(B + 1, 0), ro(B + 1, 0);
    for (int q = 0; q < Q; ++q) {
        const int b = s->q_rec[q];
        v[p.q_rec + q] = b;
        v[p.q_type + q] = s->q_type[q];
        v[p.q_span + 2 * q] = s->q_span[2 * q];
        v[p.q_span + 2 * q + 1] = s->q_span[2 * q + 1];
        ++rq[b + 1];
        ro[b + 1] += s->q_opt_off[q + 1] - s->q_opt_off[q];
        for (int j = s->q_opt_off[q]; j < s->q_opt_off[q + 1]; ++j) {
            v[p.o_rec + j] = b;
            v[p.o_q + j] = q;
        }
    }
    for (int q = 0; q <= Q; ++q) v[p.q_opt_off + q] = s->q_opt_off[q];
    for (int j = 0; j < 2 * O; ++j) v[p.o_span + j] = s->o_span[j];
    for (int b = 0; b < B; ++b) {
        rq[b + 1] += rq[b];
        ro[b + 1] += ro[b];
    }
    for (int b = 0; b <= B; ++b) {
        v[p.rec_q_off + b] = rq[b];
        v[p.rec_o_off + b] = ro[b];
        if (b < B) p.max_rec_options = std::max(p.max_rec_options, ro[b + 1] - ro[b]);
    }
    p.tile_rec = put(p.n_mtiles);
    p.tile_a_row = put(p.n_mtiles);
    {
        int m = 0;
        for (int b = 0; b < B; ++b) {
            const int nt = (s->lengths[b] + kTile - 1) / kTile;
            for (int k = 0; k < nt; ++k, ++m) {
                v[p.tile_rec + m] = b;
                v[p.tile_a_row + m] = b * s->Lpad + k * kTile;
            }
        }
    }
    p.n_items = Q + O + B;
    while (v.size() % 4) v.push_back(0);  // the item table's rows are 16-byte aligned
    p.item = put(4 * size_t(p.n_items));
    {
        // pooling work items, most rows first (option items read two rows per span row),
        // so that the last wave of CTAs holds the short ones
        std::vector<std::pair<int, int>> cost;  // (rows read, item id)
        cost.reserve(p.n_items);
        for (int q = 0; q < Q; ++q) cost.push_back({s->q_span[2 * q + 1] - s->q_span[2 * q], q});
        for (int j = 0; j < O; ++j) cost.push_back({2 * (s->o_span[2 * j + 1] - s->o_span[2 * j]), Q + j});
        for (int b = 0; b < B; ++b) cost.push_back({1, Q + O + b});
        std::stable_sort(cost.begin(), cost.end(),
                         [](const std::pair<int, int>& x, const std::pair<int, int>& y) { return x.first > y.first; });
        for (int i = 0; i < p.n_items; ++i) {
            const int id = cost[i].second;
            // one row per item: {kind << 30 | index, record, span start, span end}
            int32_t* row = &v[p.item + 4 * size_t(i)];
            if (id < Q) {
                row[0] = id;
                row[1] = s->q_rec[id];
                row[2] = s->q_span[2 * id];
                row[3] = s->q_span[2 * id + 1];
            } else if (id < Q + O) {
                const int j = id - Q;
                row[0] = (1 << 30) | j;
                row[1] = v[p.o_rec + j];
                row[2] = s->o_span[2 * j];
                row[3] = s->o_span[2 * j + 1];
            } else {
                const int b = id - Q - O;
                row[0] = (2 << 30) | b;
                row[1] = b;
                row[2] = s->lengths[b] - 1;
                row[3] = s->lengths[b];
            }
        }
    }
    p.n_chunks = nch;
    p.chunk_rec = put(nch);
    p.chunk_idx = put(nch);
    {
        int i = 0;
        for (int b = 0; b < B; ++b) {
            const int n = (s->lengths[b] + kAttnChunk - 1) / kAttnChunk;
            for (int k = 0; k < n; ++k, ++i) { v[p.chunk_rec + i] = b; v[p.chunk_idx + i] = k; }
        }
    }
    // routing-attention work units: (chunk, block of kAttnQRows options of the chunk's
    // record), chunk-major so that units working at the same time share memory rows
    {
        int n = 0;
        for (int cx = 0; cx < nch; ++cx) {
            const int b = v[p.chunk_rec + cx];
            n += (ro[b + 1] - ro[b] + kAttnQRows - 1) / kAttnQRows;
        }
        p.n_units = n;
        p.unit_cx = put(n);
        p.unit_qp = put(n);
        int u = 0;
        for (int cx = 0; cx < nch; ++cx) {
            const int b = v[p.chunk_rec + cx];
            const int nq = (ro[b + 1] - ro[b] + kAttnQRows - 1) / kAttnQRows;
            for (int qp = 0; qp < nq; ++qp, ++u) {
                v[p.unit_cx + u] = cx;
                v[p.unit_qp + u] = qp;
            }
        }
    }
    p.grp_rec = put(B + 1);    // filled by plan_tail_groups
    if (v.size() & 1) put(1);  // 8-byte alignment of the int64 table
    p.rec_part_off = put(2 * size_t(B));
    int64_t P = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t off = P;
        std::memcpy(&v[p.rec_part_off + 2 * b], &off, 8);
        const int n = (s->lengths[b] + kAttnChunk - 1) / kAttnChunk;
        P += int64_t(n) * c->heads * (ro[b + 1] - ro[b]);
    }
    p.P = P;
}

// Record groups of the fused tail: consecutive records, at most kMaxFields fields and
// kTailMaxRecOptions options per group, and about B / clusters records per group (the
// clusters the GPU holds at once), so that the groups run in one wave where the limits
// allow.
void plan_tail_groups(Plan& p, int clusters) {
    int32_t* g = &p.blob[p.grp_rec];
    const int per = clusters > 0 ? (p.B + clusters - 1) / clusters : 1;
    int n = 0, cf = 0, co = 0, cr = 0;
    g[0] = 0;
    for (int b = 0; b < p.B; ++b) {
        const int f = p.blob[p.rec_q_off + b + 1] - p.blob[p.rec_q_off + b];
        const int o = p.blob[p.rec_o_off + b + 1] - p.blob[p.rec_o_off + b];
        if (cr > 0 && (cf + f > kMaxFields || co + o > kTailMaxRecOptions || cr >= per)) {
            g[++n] = b;
            cf = co = cr = 0;
        }
        cf += f;
        co += o;
        ++cr;
    }
    g[++n] = p.B;
    p.n_groups = n;
}

// Split count of a residual-stream projection of `rows` rows (its partial products are
// summed by the LayerNorm that follows it).
int partial_splits(int rows, int N, int K) {
    int bn = 0, S = 1;
    partial_split_config((rows + kTile - 1) / kTile, N, K, &bn, &S);
    return S;
}

struct WsLayout {
    size_t flags, plan, mu, rstd, row_flags, kv, a_query, a_field, u32, x32, g32, o_res, ln_buf,
        q_buf, attn_buf, hid_buf, o_hat, f_res, f_hat, z, pm, pl, pacc, stage, part, total;
    WsLayout() = default;
    WsLayout(const clef_config* c, const Plan& p) {
        const size_t H = c->hidden, D = c->width, F = c->ffn, NKV = size_t(2) * c->n_route * D;
        const size_t B = p.B, Q = p.Q, O = p.O, R = p.R, MQO = std::max(Q, O);
        // split-K partial products of the residual-stream projections (option query,
        // routing / joint output and FFN-out projections, field projection)
        const int iD = int(D), iH = int(H), iF = int(F);
        size_t part_elems = 0;
        if (O > 0)
            for (int K : {3 * iH, iD, iF})
                part_elems = std::max(part_elems, size_t(partial_splits(int(O), iD, K)) * O * D);
        if (Q > 0)
            for (int K : {2 * iH + iD, iD, iF})
                part_elems = std::max(part_elems, size_t(partial_splits(int(Q), iD, K)) * Q * D);
        Carve cv;
        flags = cv.take(256);
        plan = cv.take(p.blob.size() * 4);
        mu = cv.take(R * 4);
        rstd = cv.take(R * 4);
        row_flags = cv.take(R / 4 * 8);  // publication flags of the statistics, one per 4 rows
        kv = cv.take(R * NKV * 2);
        a_query = cv.take(O * 3 * H * 2);
        a_field = cv.take(Q * (2 * H + D) * 2);
        u32 = cv.take(Q * H * 4);
        x32 = cv.take(O * H * 4);
        g32 = cv.take(B * H * 4);
        o_res = cv.take(O * D * 4);
        ln_buf = cv.take(MQO * D * 2);
        q_buf = cv.take(std::max(O * D, Q * 3 * D) * 2);
        attn_buf = cv.take(MQO * D * 2);
        hid_buf = cv.take(MQO * std::max(F, D) * 2);
        o_hat = cv.take(O * D * 4);
        f_res = cv.take(Q * D * 4);
        f_hat = cv.take(Q * D * 4);
        z = cv.take(O * 4 * D * 2);
        pm = cv.take(size_t(p.P) * 4);
        pl = cv.take(size_t(p.P) * 4);
        pacc = cv.take(size_t(p.P) * 64 * 4);
        stage = cv.take(size_t(kStageRows) * H * 2);  // bf16 copy of fp16 streamed rows
        part = cv.take(part_elems * 4);
        total = cv.off;
    }
};

// The validated plan and workspace layout of the schema this thread passed last.  The
// calls of one batch (workspace size, stream begin, every chunk, stream finish, forward)
// pass the same tables again and again, so each call compares them, element by element,
// with the copy kept from the previous call and validates and rebuilds only when they
// differ (or the configuration or the current device does).
struct PlanCache {
    bool valid = false;
    clef_config cfg{};
    int device = -1;
    int32_t B = 0, Lpad = 0, Q = 0, O = 0;
    int64_t row_stride = 0;
    std::vector<int32_t> tables;  // lengths | q_rec | q_type | q_span | q_opt_off | o_span
    Plan plan;
    WsLayout layout;
};

int cached_plan(const clef_config* cfg, const clef_schema* s, const Plan** plan, const WsLayout** layout) {
    thread_local PlanCache c;
    if (!s || !s->lengths || !s->q_rec || !s->q_type || !s->q_span || !s->q_opt_off || !s->o_span || s->B < 1 ||
        s->Q < 1 || s->O < 1)
        return CLEF_ERR_INVALID_ARGUMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        dev = -1;
    }
    const size_t nB = size_t(s->B), nQ = size_t(s->Q), nO = size_t(s->O);
    const std::pair<const int32_t*, size_t> parts[] = {{s->lengths, nB},     {s->q_rec, nQ},       {s->q_type, nQ},
                                                       {s->q_span, 2 * nQ},  {s->q_opt_off, nQ + 1}, {s->o_span, 2 * nO}};
    bool hit = c.valid && std::memcmp(&c.cfg, cfg, sizeof(clef_config)) == 0 && c.device == dev && c.B == s->B &&
               c.Lpad == s->Lpad && c.Q == s->Q && c.O == s->O && c.row_stride == s->row_stride;
    if (hit) {
        size_t off = 0;
        for (const auto& pt : parts) {
            if (std::memcmp(c.tables.data() + off, pt.first, pt.second * sizeof(int32_t)) != 0) {
                hit = false;
                break;
            }
            off += pt.second;
        }
    }
    if (!hit) {
        c.valid = false;
        const int v = validate_schema(cfg, s);
        if (v != CLEF_OK) return v;
        c.plan = Plan();
        build_plan(cfg, s, c.plan);
        plan_tail_groups(c.plan, record_tail_clusters());
        c.layout = WsLayout(cfg, c.plan);
        c.tables.clear();
        for (const auto& pt : parts) c.tables.insert(c.tables.end(), pt.first, pt.first + pt.second);
        c.cfg = *cfg;
        c.device = dev;
        c.B = s->B;
        c.Lpad = s->Lpad;
        c.Q = s->Q;
        c.O = s->O;
        c.row_stride = s->row_stride;
        c.valid = true;
    }
    *plan = &c.plan;
    *layout = &c.layout;
    return CLEF_OK;
}

// Clears the workspace status word (and, when given, the statistics' publication
// flags) and uploads the plan, all asynchronously on `st`.  The status word therefore
// reports the device-side errors of the latest call.
int upload_plan(const Plan& p, void* workspace, void* dst, cudaStream_t st, void* row_flags = nullptr,
                size_t row_flags_bytes = 0) {
    if (launch_plan_upload(static_cast<int32_t*>(dst), p.blob.data(), p.blob.size(), workspace, 256, row_flags,
                           row_flags ? row_flags_bytes : 0, st) != cudaSuccess)
        return CLEF_ERR_CUDA;
    return CLEF_OK;
}

#define CK(x)                                   \
    do {                                        \
        if ((x) != cudaSuccess) return CLEF_ERR_CUDA; \
    } while (0)

inline const uint16_t* W(const void* const* w, int i) { return static_cast<const uint16_t*>(w[i]); }

inline cudaError_t mark(const clef_debug_outputs* d, int slot, cudaStream_t st) {
    if (!d || !d->events[slot]) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(d->events[slot]), st);
}

// Dense GEMM helper: A [M][K] (lda), weight [N][K]; K may be split across a cluster.
cudaError_t dense(const uint16_t* A, int64_t lda, int M, const uint16_t* Bw, int N, int K, const GemmEpilogue& e,
                  int* flags, cudaStream_t st) {
    GemmProblem g;
    g.allow_split = true;
    g.b_is_weight = true;
    g.A = A;
    g.lda = lda;
    g.a_rows = M;
    g.B = Bw;
    g.ldb = K;
    g.N = N;
    g.K = K;
    g.n_mtiles = (M + kTile - 1) / kTile;
    GemmEpilogue ee = e;
    ee.M = M;
    return launch_gemm(g, ee, flags, st);
}

// Residual-stream projection A [M][K] x weight [N][K]^T whose K is split over
// independent CTAs; each split stores its fp32 partial product into its slab of `part`
// (slab stride M * N) and the LayerNorm that follows sums them (launch_layer_norm_acc).
cudaError_t dense_partial(const uint16_t* A, int64_t lda, int M, const uint16_t* Bw, int N, int K, float* part,
                          int* flags, cudaStream_t st, int* splits) {
    int bn = 0, S = 1;
    partial_split_config((M + kTile - 1) / kTile, N, K, &bn, &S);
    *splits = S;
    GemmProblem g;
    g.b_is_weight = true;
    g.A = A;
    g.lda = lda;
    g.a_rows = M;
    g.B = Bw;
    g.ldb = K;
    g.N = N;
    g.K = K;
    g.n_mtiles = (M + kTile - 1) / kTile;
    g.defer_splits = S;
    g.defer_bn = bn;
    g.part_stride = int64_t(M) * N;
    GemmEpilogue e;
    e.kind = EPI_F32;
    e.out = part;
    e.ldo = N;
    e.M = M;
    return launch_gemm(g, e, flags, st);
}

}  // namespace

extern "C" {

const char* clef_status_string(int s) {
    switch (s) {
        case CLEF_OK: return "ok";
        case CLEF_ERR_INVALID_ARGUMENT: return "invalid argument";
        case CLEF_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case CLEF_ERR_UNSUPPORTED_CONFIG: return "unsupported configuration";
        case CLEF_ERR_CUDA: return "CUDA error";
        case CLEF_ERR_DEVICE_BOUNDS: return "device-side index out of range";
        case CLEF_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

int clef_weight_count(const clef_config* cfg) {
    if (!config_ok(cfg)) return -1;
    return WIdx(cfg).count();
}

int clef_prepared_size(const clef_config* cfg, size_t* bytes) {
    if (!bytes) return CLEF_ERR_INVALID_ARGUMENT;
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    *bytes = PreparedLayout(cfg).total;
    return CLEF_OK;
}

int clef_prepare_weights(const clef_config* cfg, const void* const* weights, void* prepared, size_t prepared_bytes,
                         void* stream) {
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    if (!weights || !prepared || (reinterpret_cast<uintptr_t>(prepared) & 255)) return CLEF_ERR_INVALID_ARGUMENT;
    const WIdx wi(cfg);
    for (int i = 0; i < wi.count(); ++i)
        if (!weights[i] || (reinterpret_cast<uintptr_t>(weights[i]) & 15)) return CLEF_ERR_INVALID_ARGUMENT;
    const PreparedLayout L(cfg);
    if (prepared_bytes < L.total) return CLEF_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(prepared);
    const int H = cfg->hidden, D = cfg->width;
    FoldArgs f;
    f.H = H;
    f.D = D;
    for (int l = 0; l < cfg->n_route; ++l) {
        f.w[2 * l] = W(weights, wi.route(l, 4));
        f.bias[2 * l] = W(weights, wi.route(l, 5));
        f.w[2 * l + 1] = W(weights, wi.route(l, 6));
        f.bias[2 * l + 1] = W(weights, wi.route(l, 7));
    }
    f.gamma = W(weights, 0);
    f.beta = W(weights, 1);
    f.out_w = reinterpret_cast<uint16_t*>(base + L.wkv);
    f.out_c = reinterpret_cast<float*>(base + L.ckv);
    f.out_b = reinterpret_cast<float*>(base + L.bkv);
    CK(launch_fold_kv(f, 2 * cfg->n_route * D, st));
    uint16_t* wq0 = reinterpret_cast<uint16_t*>(base + L.wq0);
    CK(launch_copy_cols(wq0, 3 * H, 0, W(weights, 2), H, D, H, st));
    CK(launch_copy_cols(wq0, 3 * H, H, W(weights, 3), H, D, H, st));
    CK(launch_copy_cols(wq0, 3 * H, 2 * H, W(weights, 4), H, D, H, st));
    uint16_t* wf = reinterpret_cast<uint16_t*>(base + L.wfield);
    const int ldf = 2 * H + D;
    CK(launch_copy_cols(wf, ldf, 0, W(weights, wi.mid(4)), H, D, H, st));
    CK(launch_copy_cols(wf, ldf, H, W(weights, wi.mid(6)), H, D, H, st));
    CK(launch_copy_cols(wf, ldf, 2 * H, W(weights, wi.mid(5)), D, D, D, st));
    if (L.tail) {  // the fused tail's weight rows, sliced per cluster CTA
        auto dst = [&](size_t off) { return reinterpret_cast<uint16_t*>(base + off); };
        const int F = cfg->ffn, CT = cfg->heads;  // cluster CTAs: one per head
        CK(launch_tail_slices(wf, ldf, D / CT, 0, D, dst(L.t_field), st));
        CK(launch_tail_slices(W(weights, wi.tail(4)), 4 * D, D / CT, 0, D, dst(L.t_mlp1), st));
        for (int i = 0; i < cfg->n_joint; ++i) {
            CK(launch_tail_slices(W(weights, wi.joint(i, 2)), D, 3 * D / CT, 1, D, dst(L.t_qkv[i]), st));
            CK(launch_tail_slices(W(weights, wi.joint(i, 4)), D, D / CT, 0, D, dst(L.t_o[i]), st));
            CK(launch_tail_slices(W(weights, wi.joint(i, 8)), D, F / CT, 0, D, dst(L.t_w1[i]), st));
            CK(launch_tail_slices(W(weights, wi.joint(i, 10)), F, D / CT, 0, D, dst(L.t_w2[i]), st));
        }
    }
    return CLEF_OK;
}

int clef_workspace_size(const clef_config* cfg, const clef_schema* schema, size_t* bytes) {
    if (!bytes) return CLEF_ERR_INVALID_ARGUMENT;
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    const Plan* pp = nullptr;
    const WsLayout* lp = nullptr;
    const int v = cached_plan(cfg, schema, &pp, &lp);
    if (v != CLEF_OK) return v;
    *bytes = lp->total;
    return CLEF_OK;
}

}  // extern "C"

namespace {

enum ForwardMode { kForwardFull = 0, kForwardAfterStream = 1 };

// The per-record tail (option LayerNorm to softmax) has two implementations.  The
// batched chain runs every projection as one GEMM over the whole batch, so each weight
// matrix is streamed once, by up to every SM.  The fused launch (record_tail.cu) runs
// one 16-CTA cluster per record group and saves ~30 launches, but each cluster CTA
// streams its slice of every weight matrix itself (7.7 MB per CTA at the pages' head
// shape), at the ~60-120 GB/s one SM takes in.  Measured on GB300 the batched chain is
// faster for every workload tried (batch8_l16k 3.32 vs 3.52 ms per forward, the 1-record
// reference 0.405 vs 0.417 ms), so it is the default; debug->tail_mode = 2 selects the
// fused launch where the head shape allows it (width 1024, 16 heads, FFN 4096, at most
// kTailMaxRecOptions options per record).
bool use_record_tail(const clef_config* c, const Plan& p, const clef_debug_outputs* debug) {
    if (!debug || debug->tail_mode != 2) return false;
    if (!record_tail_shape(c->hidden, c->width, c->heads, c->ffn, c->n_joint)) return false;
    if (p.max_rec_options > kTailMaxRecOptions) return false;
    return record_tail_clusters() > 0;
}

// Debug copies and the launch count, after the last kernel of the forward pass.
int finish_debug(const clef_debug_outputs* debug, int n_launch, int Q, int O, int B, int H, int D, const float* u32,
                 const float* x32, const float* g32, const float* o_hat, const float* f_hat, const float* mu,
                 const float* rstd, int R, cudaStream_t st) {
    if (!debug) return CLEF_OK;
    if (debug->row_mu) CK(cudaMemcpyAsync(debug->row_mu, mu, size_t(R) * 4, cudaMemcpyDeviceToDevice, st));
    if (debug->row_rstd) CK(cudaMemcpyAsync(debug->row_rstd, rstd, size_t(R) * 4, cudaMemcpyDeviceToDevice, st));
    if (debug->timeline_count) CK(cudaMemcpyAsync(debug->timeline_count, &n_launch, 4, cudaMemcpyHostToDevice, st));
    if (debug->pooled_u) CK(cudaMemcpyAsync(debug->pooled_u, u32, size_t(Q) * H * 4, cudaMemcpyDeviceToDevice, st));
    if (debug->pooled_x) CK(cudaMemcpyAsync(debug->pooled_x, x32, size_t(O) * H * 4, cudaMemcpyDeviceToDevice, st));
    if (debug->global_g) CK(cudaMemcpyAsync(debug->global_g, g32, size_t(B) * H * 4, cudaMemcpyDeviceToDevice, st));
    if (debug->option_final)
        CK(cudaMemcpyAsync(debug->option_final, o_hat, size_t(O) * D * 4, cudaMemcpyDeviceToDevice, st));
    if (debug->field_final)
        CK(cudaMemcpyAsync(debug->field_final, f_hat, size_t(Q) * D * 4, cudaMemcpyDeviceToDevice, st));
    return CLEF_OK;
}

// The forward pass.  kForwardFull uploads the plan and computes the memory statistics
// and K/V itself; kForwardAfterStream finds both already in the workspace (put there by
// clef_stream_begin / clef_stream_rows) and only zeroes the records' round-up slack rows.
int forward_impl(const clef_config* cfg, const void* const* weights, const void* prepared,
                 const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                 const uint16_t* lexical, float* logits, float* probs, float* q_value, float* q_conf,
                 int32_t* q_argmax, void* workspace, size_t workspace_bytes, const clef_debug_outputs* debug,
                 void* stream, int mode, bool hidden_f16 = false) {
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    if (hidden_f16 && mode != kForwardAfterStream) return CLEF_ERR_INVALID_ARGUMENT;
    if (!weights || !prepared || !hidden || !token_ids || !lexical || !logits || !probs || !q_value || !q_conf ||
        !q_argmax || !workspace)
        return CLEF_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(lexical) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(prepared) & 255))
        return CLEF_ERR_INVALID_ARGUMENT;
    const WIdx wi(cfg);
    for (int i = 0; i < wi.count(); ++i)
        if (!weights[i] || (reinterpret_cast<uintptr_t>(weights[i]) & 15)) return CLEF_ERR_INVALID_ARGUMENT;
    const Plan* pp = nullptr;
    const WsLayout* lp = nullptr;
    const int v = cached_plan(cfg, schema, &pp, &lp);
    if (v != CLEF_OK) return v;
    const Plan& p = *pp;
    const WsLayout& L = *lp;
    if (workspace_bytes < L.total) return CLEF_ERR_WORKSPACE_TOO_SMALL;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int n_launch = 0;
    // records the next timeline event (if asked for) after a launch
    auto tick = [&]() -> cudaError_t {
        const int k = n_launch++;
        if (!debug || !debug->timeline || k >= debug->timeline_len || !debug->timeline[k]) return cudaSuccess;
        return cudaEventRecord(static_cast<cudaEvent_t>(debug->timeline[k]), st);
    };
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* pw = static_cast<const uint8_t*>(prepared);
    const PreparedLayout PL(cfg);
    int* flags = reinterpret_cast<int*>(ws + L.flags);
    const int32_t* plan = reinterpret_cast<const int32_t*>(ws + L.plan);
    const int H = cfg->hidden, D = cfg->width, F = cfg->ffn, NKV = 2 * cfg->n_route * D;
    const int B = p.B, Q = p.Q, O = p.O;

    if (mode == kForwardFull) {
        const int u = upload_plan(p, ws, ws + L.plan, st, ws + L.row_flags, size_t(p.R) / 4 * 8);
        if (u != CLEF_OK) return u;
    }
    auto T = [&](size_t off) { return plan + off; };
    float* mu = reinterpret_cast<float*>(ws + L.mu);
    float* rstd = reinterpret_cast<float*>(ws + L.rstd);
    uint16_t* kv = reinterpret_cast<uint16_t*>(ws + L.kv);
    uint16_t* a_query = reinterpret_cast<uint16_t*>(ws + L.a_query);
    uint16_t* a_field = reinterpret_cast<uint16_t*>(ws + L.a_field);
    float* u32 = reinterpret_cast<float*>(ws + L.u32);
    float* x32 = reinterpret_cast<float*>(ws + L.x32);
    float* g32 = reinterpret_cast<float*>(ws + L.g32);
    float* o_res = reinterpret_cast<float*>(ws + L.o_res);
    uint16_t* ln_buf = reinterpret_cast<uint16_t*>(ws + L.ln_buf);
    uint16_t* q_buf = reinterpret_cast<uint16_t*>(ws + L.q_buf);
    uint16_t* attn_buf = reinterpret_cast<uint16_t*>(ws + L.attn_buf);
    uint16_t* hid_buf = reinterpret_cast<uint16_t*>(ws + L.hid_buf);
    float* o_hat = reinterpret_cast<float*>(ws + L.o_hat);
    float* f_res = reinterpret_cast<float*>(ws + L.f_res);
    float* f_hat = reinterpret_cast<float*>(ws + L.f_hat);
    uint16_t* z = reinterpret_cast<uint16_t*>(ws + L.z);
    float* part = reinterpret_cast<float*>(ws + L.part);
    const int ld_field = 2 * H + D;
    // the stream update + LayerNorm that finishes a deferred split-K projection
    auto ln_acc = [&](float* x, int rows, int S, const uint16_t* bias, bool resid, const uint16_t* ln_w,
                      const uint16_t* ln_b, uint16_t* out_bf16, float* out_f32, const uint16_t* table = nullptr,
                      const int32_t* idx = nullptr) {
        LnAccArgs la;
        la.x = x; la.rows = rows; la.D = D; la.part = part; la.part_stride = int64_t(rows) * D; la.S = S;
        la.bias = bias; la.row_table = table; la.row_idx = idx; la.ld_table = D; la.resid = resid ? 1 : 0;
        la.ln_w = ln_w; la.ln_b = ln_b; la.out_bf16 = out_bf16; la.out_f32 = out_f32;
        return launch_layer_norm_acc(la, st);
    };
    int splits = 1;

    // 1. memory K/V of every routing layer (LayerNorm folded), real rows only; the
    // projection also writes the memory row statistics that pooling applies the memory
    // LayerNorm through
    if (mode == kForwardAfterStream) {
        // K/V rows and statistics came in chunk by chunk; the round-up slack rows of each
        // record were never written, and attention reads whole tiles, so they are zeroed here
        CK(launch_zero_slack(kv, NKV, T(p.rec_row_off), T(p.lengths), B, st)); CK(tick());
    } else {
        GemmProblem g;
        g.A = hidden; g.lda = schema->row_stride; g.a_rows = int64_t(B) * schema->Lpad;
        g.B = reinterpret_cast<const uint16_t*>(pw + PL.wkv); g.ldb = H;
        g.N = NKV; g.K = H; g.n_mtiles = p.n_mtiles; g.a_row_of_mtile = T(p.tile_a_row);
        GemmEpilogue e;
        e.kind = EPI_KV_LNFOLD; e.row_mu = mu; e.row_rstd = rstd;
        e.tile_rec = T(p.tile_rec); e.rec_row_off = T(p.rec_row_off); e.rec_len = T(p.lengths);
        e.row_flags = reinterpret_cast<uint64_t*>(ws + L.row_flags);
        e.col_c = reinterpret_cast<const float*>(pw + PL.ckv);
        e.bias_f32 = reinterpret_cast<const float*>(pw + PL.bkv);
        e.out = kv; e.ldo = NKV; e.M = p.R;
        CK(mark(debug, 0, st));
        CK(launch_gemm(g, e, flags, st)); CK(tick());
        CK(mark(debug, 1, st));
    }
    // 2. span pooling
    SpanPoolArgs sp{};
    sp.hidden = hidden; sp.row_stride = schema->row_stride; sp.Lpad = schema->Lpad; sp.H = H; sp.vocab = cfg->vocab;
    sp.token_ids = token_ids; sp.lexical = lexical; sp.mu = mu; sp.rstd = rstd;
    sp.ln_w = W(weights, 0); sp.ln_b = W(weights, 1);
    sp.items = reinterpret_cast<const int4*>(T(p.item));
    sp.lengths = T(p.lengths); sp.rec_row_off = T(p.rec_row_off); sp.rec_q_off = T(p.rec_q_off);
    sp.q_rec = T(p.q_rec); sp.q_span = T(p.q_span); sp.q_opt_off = T(p.q_opt_off);
    sp.o_rec = T(p.o_rec); sp.o_span = T(p.o_span);
    sp.a_query = a_query; sp.ld_query = 3 * H; sp.a_field = a_field; sp.ld_field = ld_field;
    sp.u32 = u32; sp.x32 = x32; sp.g32 = g32;
    sp.dbg_c = debug ? debug->pooled_c : nullptr;
    sp.flags = flags;
    sp.in_f16 = hidden_f16 ? 1 : 0;
    CK(mark(debug, 4, st));
    CK(launch_span_pool(sp, p.n_items, false, st)); CK(tick());
    CK(mark(debug, 5, st));
    // 3. option queries: o = [c | x | u] [W_ctx | W_lex | W_qst]^T + b (the sum of the
    // split partial products and the bias is formed by the first routing LayerNorm)
    CK(dense_partial(a_query, 3 * H, O, reinterpret_cast<const uint16_t*>(pw + PL.wq0), D, 3 * H, part, flags, st,
                     &splits)); CK(tick());
    const uint16_t* pending_bias = W(weights, 5);  // bias of the projection whose partials are in `part`
    bool pending_resid = false;
    // 5. evidence routing layers
    RouteAttnArgs ra{};
    ra.q = q_buf; ra.ldq = D; ra.kv = kv; ra.ldkv = NKV; ra.kv_rows = p.R; ra.heads = cfg->heads; ra.flags = flags;
    ra.scale_log2 = 1.4426950408889634f / 8.0f;
    ra.chunk_rec = T(p.chunk_rec); ra.chunk_idx = T(p.chunk_idx); ra.lengths = T(p.lengths);
    ra.unit_cx = T(p.unit_cx); ra.unit_qp = T(p.unit_qp); ra.n_units = p.n_units;
    ra.rec_row_off = T(p.rec_row_off); ra.rec_o_off = T(p.rec_o_off);
    ra.rec_part_off = reinterpret_cast<const int64_t*>(T(p.rec_part_off)); ra.o_rec = T(p.o_rec);
    ra.pm = reinterpret_cast<float*>(ws + L.pm); ra.pl = reinterpret_cast<float*>(ws + L.pl);
    ra.pacc = reinterpret_cast<float*>(ws + L.pacc); ra.out = attn_buf; ra.ldo = D;
    for (int l = 0; l < cfg->n_route; ++l) {
        CK(ln_acc(o_res, O, splits, pending_bias, pending_resid, W(weights, wi.route(l, 0)), W(weights, wi.route(l, 1)),
                  ln_buf, nullptr)); CK(tick());
        GemmEpilogue eq;
        eq.kind = EPI_BF16; eq.bias_bf16 = W(weights, wi.route(l, 3)); eq.out = q_buf; eq.ldo = D;
        CK(dense(ln_buf, D, O, W(weights, wi.route(l, 2)), D, D, eq, flags, st)); CK(tick());
        ra.k_col = 2 * l * D;
        ra.v_col = (2 * l + 1) * D;
        if (l == 0) CK(mark(debug, 2, st));
        CK(launch_route_attn_partial(ra, O, st)); CK(tick());
        if (l == 0) CK(mark(debug, 3, st));
        CK(launch_route_attn_merge(ra, O, st)); CK(tick());
        CK(dense_partial(attn_buf, D, O, W(weights, wi.route(l, 8)), D, D, part, flags, st, &splits)); CK(tick());
        CK(ln_acc(o_res, O, splits, W(weights, wi.route(l, 9)), true, W(weights, wi.route(l, 10)),
                  W(weights, wi.route(l, 11)), ln_buf, nullptr)); CK(tick());
        GemmEpilogue e1;
        e1.kind = EPI_BF16; e1.gelu = 1; e1.bias_bf16 = W(weights, wi.route(l, 13)); e1.out = hid_buf; e1.ldo = F;
        CK(dense(ln_buf, D, O, W(weights, wi.route(l, 12)), F, D, e1, flags, st)); CK(tick());
        CK(dense_partial(hid_buf, F, O, W(weights, wi.route(l, 14)), D, F, part, flags, st, &splits)); CK(tick());
        pending_bias = W(weights, wi.route(l, 15));
        pending_resid = true;
    }
    // the option stream's last projection finished, then the final option LayerNorm
    CK(ln_acc(o_res, O, splits, pending_bias, pending_resid, W(weights, wi.mid(0)), W(weights, wi.mid(1)), nullptr,
              o_hat)); CK(tick());
    // 6-8. the per-record tail: one cluster launch per batch when it applies (see
    // use_record_tail), else the batched chain below
    if (use_record_tail(cfg, p, debug)) {
        RecordTailArgs rt{};
        rt.B = B; rt.H = H; rt.D = D; rt.F = F; rt.n_joint = cfg->n_joint; rt.Q = Q; rt.O = O;
        rt.n_groups = p.n_groups; rt.grp_rec = T(p.grp_rec); rt.flags = flags;
        rt.rec_q_off = T(p.rec_q_off); rt.rec_o_off = T(p.rec_o_off); rt.q_type = T(p.q_type); rt.q_rec = T(p.q_rec);
        rt.q_opt_off = T(p.q_opt_off); rt.o_q = T(p.o_q);
        rt.o_res = o_res; rt.u32 = u32; rt.g32 = g32; rt.x32 = x32; rt.a_field = a_field; rt.ld_field = ld_field;
        rt.opt_ln_w = W(weights, wi.mid(0)); rt.opt_ln_b = W(weights, wi.mid(1));
        rt.pool_w = W(weights, wi.mid(2)); rt.pool_b = W(weights, wi.mid(3));
        auto sl = [&](size_t off) { return reinterpret_cast<const uint16_t*>(pw + off); };
        rt.w_field = sl(PL.t_field); rt.b_field = W(weights, wi.mid(7));
        rt.type_emb = W(weights, wi.mid(8));
        for (int i = 0; i < cfg->n_joint; ++i) {
            rt.ln1_w[i] = W(weights, wi.joint(i, 0)); rt.ln1_b[i] = W(weights, wi.joint(i, 1));
            rt.w_qkv[i] = sl(PL.t_qkv[i]); rt.b_qkv[i] = W(weights, wi.joint(i, 3));
            rt.w_o[i] = sl(PL.t_o[i]); rt.b_o[i] = W(weights, wi.joint(i, 5));
            rt.ln2_w[i] = W(weights, wi.joint(i, 6)); rt.ln2_b[i] = W(weights, wi.joint(i, 7));
            rt.w_1[i] = sl(PL.t_w1[i]); rt.b_1[i] = W(weights, wi.joint(i, 9));
            rt.w_2[i] = sl(PL.t_w2[i]); rt.b_2[i] = W(weights, wi.joint(i, 11));
        }
        rt.fld_ln_w = W(weights, wi.tail(0)); rt.fld_ln_b = W(weights, wi.tail(1));
        rt.gate = W(weights, wi.tail(2)); rt.joint_scale = W(weights, wi.tail(3));
        rt.mlp1_w = sl(PL.t_mlp1); rt.mlp1_b = W(weights, wi.tail(5));
        rt.mlp2_w = W(weights, wi.tail(6)); rt.mlp2_b = W(weights, wi.tail(7));
        rt.o_hat = o_hat; rt.f_hat = f_hat; rt.ln_buf = ln_buf; rt.attn_buf = attn_buf; rt.hid_buf = hid_buf; rt.z = z;
        rt.logits = logits; rt.probs = probs; rt.q_value = q_value; rt.q_conf = q_conf; rt.q_argmax = q_argmax;
        CK(launch_record_tail(rt, st)); CK(tick());
        return finish_debug(debug, n_launch, Q, O, B, H, D, u32, x32, g32, o_hat, f_hat, mu, rstd, p.R, st);
    }
    // 6. fields: [u | g | summary] [W_fu | W_fg | W_fs]^T + b + type embedding (bias and
    // type-embedding row added with the partial products by the first joint LayerNorm)
    CK(launch_field_pool(o_hat, D, T(p.q_opt_off), Q, W(weights, wi.mid(2)), W(weights, wi.mid(3)), a_field, ld_field,
                         2 * H, st)); CK(tick());
    CK(dense_partial(a_field, ld_field, Q, reinterpret_cast<const uint16_t*>(pw + PL.wfield), D, ld_field, part, flags,
                     st, &splits)); CK(tick());
    pending_bias = W(weights, wi.mid(7));
    pending_resid = false;
    const uint16_t* pending_table = W(weights, wi.mid(8));
    // 7. joint layers over each record's fields
    for (int i = 0; i < cfg->n_joint; ++i) {
        CK(ln_acc(f_res, Q, splits, pending_bias, pending_resid, W(weights, wi.joint(i, 0)), W(weights, wi.joint(i, 1)),
                  ln_buf, nullptr, pending_table, T(p.q_type))); CK(tick());
        pending_table = nullptr;
        GemmEpilogue eq;
        eq.kind = EPI_BF16; eq.bias_bf16 = W(weights, wi.joint(i, 3)); eq.out = q_buf; eq.ldo = 3 * D;
        CK(dense(ln_buf, D, Q, W(weights, wi.joint(i, 2)), 3 * D, D, eq, flags, st)); CK(tick());
        CK(launch_field_attn(q_buf, D, cfg->heads, T(p.rec_q_off), B, 0.125f, attn_buf, st)); CK(tick());
        CK(dense_partial(attn_buf, D, Q, W(weights, wi.joint(i, 4)), D, D, part, flags, st, &splits)); CK(tick());
        CK(ln_acc(f_res, Q, splits, W(weights, wi.joint(i, 5)), true, W(weights, wi.joint(i, 6)),
                  W(weights, wi.joint(i, 7)), ln_buf, nullptr)); CK(tick());
        GemmEpilogue e1;
        e1.kind = EPI_BF16; e1.gelu = 1; e1.bias_bf16 = W(weights, wi.joint(i, 9)); e1.out = hid_buf; e1.ldo = F;
        CK(dense(ln_buf, D, Q, W(weights, wi.joint(i, 8)), F, D, e1, flags, st)); CK(tick());
        CK(dense_partial(hid_buf, F, Q, W(weights, wi.joint(i, 10)), D, F, part, flags, st, &splits)); CK(tick());
        pending_bias = W(weights, wi.joint(i, 11));
        pending_resid = true;
    }
    // the field stream's last projection finished, the final field LayerNorm, and the scorer
    // MLP input z_j = [f_hat_q, o_hat_j, f_hat_q * o_hat_j, |f_hat_q - o_hat_j|] of each option
    {
        LnAccArgs la;
        la.x = f_res; la.rows = Q; la.D = D; la.part = part; la.part_stride = int64_t(Q) * D; la.S = splits;
        la.bias = pending_bias; la.row_table = pending_table; la.row_idx = T(p.q_type); la.ld_table = D;
        la.resid = pending_resid ? 1 : 0; la.ln_w = W(weights, wi.tail(0)); la.ln_b = W(weights, wi.tail(1));
        la.out_f32 = f_hat; la.z = z; la.z_opt_off = T(p.q_opt_off); la.z_o_hat = o_hat;
        CK(launch_layer_norm_acc(la, st)); CK(tick());
    }
    // 8. scorer MLP hidden layer, then scores, softmax and answers
    {
        GemmEpilogue e;
        e.kind = EPI_BF16; e.gelu = 1; e.bias_bf16 = W(weights, wi.tail(5)); e.out = hid_buf; e.ldo = D;
        CK(dense(z, 4 * D, O, W(weights, wi.tail(4)), D, 4 * D, e, flags, st)); CK(tick());
    }
    ScoreArgs sc{};
    sc.H = H; sc.D = D; sc.q_rec = T(p.q_rec); sc.q_type = T(p.q_type); sc.q_opt_off = T(p.q_opt_off);
    sc.u32 = u32; sc.g32 = g32; sc.x32 = x32; sc.f_hat = f_hat; sc.o_hat = o_hat; sc.mlp_hidden = hid_buf;
    sc.w2 = W(weights, wi.tail(6)); sc.b2 = W(weights, wi.tail(7)); sc.gate = W(weights, wi.tail(2));
    sc.joint_scale = W(weights, wi.tail(3));
    sc.logits = logits; sc.probs = probs; sc.q_value = q_value; sc.q_conf = q_conf; sc.q_argmax = q_argmax;
    CK(launch_score_softmax(sc, Q, st)); CK(tick());
    return finish_debug(debug, n_launch, Q, O, B, H, D, u32, x32, g32, o_hat, f_hat, mu, rstd, p.R, st);
}

// Statistics and K/V of rows [row0, row0 + n_rows) of one record.  fp16 rows are first
// rounded to bf16 into the workspace staging area, kStageRows at a time; the projection
// (which computes the statistics from the rows it stages) then reads that copy, exactly
// as it reads bf16 rows.
int stream_rows_impl(const clef_config* cfg, const void* prepared, const clef_schema* schema, const uint16_t* hidden,
                     int32_t record, int32_t row0, int32_t n_rows, void* workspace, size_t workspace_bytes,
                     void* stream, bool f16) {
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    if (!prepared || !hidden || !workspace || (reinterpret_cast<uintptr_t>(hidden) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(prepared) & 255))
        return CLEF_ERR_INVALID_ARGUMENT;
    const Plan* pp = nullptr;
    const WsLayout* lp = nullptr;
    const int v = cached_plan(cfg, schema, &pp, &lp);
    if (v != CLEF_OK) return v;
    if (record < 0 || record >= schema->B || row0 < 0 || n_rows < 1 ||
        int64_t(row0) + n_rows > schema->lengths[record])
        return CLEF_ERR_INVALID_ARGUMENT;
    const Plan& p = *pp;
    const WsLayout& L = *lp;
    if (workspace_bytes < L.total) return CLEF_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* pw = static_cast<const uint8_t*>(prepared);
    const PreparedLayout PL(cfg);
    const int H = cfg->hidden, NKV = 2 * cfg->n_route * cfg->width;
    const int64_t out_row0 = p.blob[p.rec_row_off + record] + int64_t(row0);  // compact row of the first row
    const uint16_t* rows0 = hidden + (int64_t(record) * schema->Lpad + row0) * schema->row_stride;
    uint16_t* stage = reinterpret_cast<uint16_t*>(ws + L.stage);
    for (int done = 0; done < n_rows;) {
        const int n = f16 ? std::min(n_rows - done, kStageRows) : n_rows;
        const uint16_t* rows = rows0 + int64_t(done) * schema->row_stride;
        int64_t ld = schema->row_stride;
        if (f16) {
            CK(launch_f16_rows_to_bf16(rows, ld, n, H, stage, st));
            rows = stage;
            ld = H;
        }
        const int64_t out_row = out_row0 + done;
        float* mu = reinterpret_cast<float*>(ws + L.mu) + out_row;
        float* rstd = reinterpret_cast<float*>(ws + L.rstd) + out_row;
        GemmProblem g;
        g.A = rows; g.lda = ld; g.a_rows = n;
        g.B = reinterpret_cast<const uint16_t*>(pw + PL.wkv); g.ldb = H;
        g.N = NKV; g.K = H; g.n_mtiles = (n + kTile - 1) / kTile;
        GemmEpilogue e;
        e.kind = EPI_KV_LNFOLD; e.row_mu = mu; e.row_rstd = rstd;
        e.row_flags = reinterpret_cast<uint64_t*>(ws + L.row_flags);  // rows of this call's tiles
        e.col_c = reinterpret_cast<const float*>(pw + PL.ckv);
        e.bias_f32 = reinterpret_cast<const float*>(pw + PL.bkv);
        e.out = reinterpret_cast<uint16_t*>(ws + L.kv) + out_row * NKV; e.ldo = NKV; e.M = n;
        CK(launch_gemm(g, e, reinterpret_cast<int*>(ws + L.flags), st));
        done += n;
    }
    return CLEF_OK;
}

}  // namespace

extern "C" {

int clef_head_forward(const clef_config* cfg, const void* const* weights, const void* prepared,
                      const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                      const uint16_t* lexical, float* logits, float* probs, float* q_value, float* q_conf,
                      int32_t* q_argmax, void* workspace, size_t workspace_bytes, const clef_debug_outputs* debug,
                      void* stream) {
    return forward_impl(cfg, weights, prepared, schema, hidden, token_ids, lexical, logits, probs, q_value, q_conf,
                        q_argmax, workspace, workspace_bytes, debug, stream, kForwardFull);
}

int clef_stream_begin(const clef_config* cfg, const clef_schema* schema, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return CLEF_ERR_INVALID_ARGUMENT;
    const Plan* pp = nullptr;
    const WsLayout* lp = nullptr;
    const int v = cached_plan(cfg, schema, &pp, &lp);
    if (v != CLEF_OK) return v;
    if (workspace_bytes < lp->total) return CLEF_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return upload_plan(*pp, ws, ws + lp->plan, static_cast<cudaStream_t>(stream), ws + lp->row_flags,
                       size_t(pp->R) / 4 * 8);
}

int clef_stream_rows(const clef_config* cfg, const void* prepared, const clef_schema* schema, const uint16_t* hidden,
                     int32_t record, int32_t row0, int32_t n_rows, void* workspace, size_t workspace_bytes,
                     void* stream) {
    return stream_rows_impl(cfg, prepared, schema, hidden, record, row0, n_rows, workspace, workspace_bytes, stream,
                            false);
}

int clef_stream_rows_f16(const clef_config* cfg, const void* prepared, const clef_schema* schema,
                         const uint16_t* hidden, int32_t record, int32_t row0, int32_t n_rows, void* workspace,
                         size_t workspace_bytes, void* stream) {
    return stream_rows_impl(cfg, prepared, schema, hidden, record, row0, n_rows, workspace, workspace_bytes, stream,
                            true);
}

int clef_stream_finish(const clef_config* cfg, const void* const* weights, const void* prepared,
                       const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                       const uint16_t* lexical, float* logits, float* probs, float* q_value, float* q_conf,
                       int32_t* q_argmax, void* workspace, size_t workspace_bytes, const clef_debug_outputs* debug,
                       void* stream) {
    return forward_impl(cfg, weights, prepared, schema, hidden, token_ids, lexical, logits, probs, q_value, q_conf,
                        q_argmax, workspace, workspace_bytes, debug, stream, kForwardAfterStream);
}

int clef_stream_finish_f16(const clef_config* cfg, const void* const* weights, const void* prepared,
                           const clef_schema* schema, const uint16_t* hidden, const int32_t* token_ids,
                           const uint16_t* lexical, float* logits, float* probs, float* q_value, float* q_conf,
                           int32_t* q_argmax, void* workspace, size_t workspace_bytes,
                           const clef_debug_outputs* debug, void* stream) {
    return forward_impl(cfg, weights, prepared, schema, hidden, token_ids, lexical, logits, probs, q_value, q_conf,
                        q_argmax, workspace, workspace_bytes, debug, stream, kForwardAfterStream, true);
}

int clef_device_status(void* workspace, void* stream) {
    if (!workspace) return CLEF_ERR_INVALID_ARGUMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int h = 0;
    CK(cudaMemcpyAsync(&h, workspace, 4, cudaMemcpyDeviceToHost, st));
    CK(cudaStreamSynchronize(st));
    if (h != 0) CK(cudaMemsetAsync(workspace, 0, 4, st));
    if (h & kFlagTimeout) return CLEF_ERR_DEVICE_TIMEOUT;
    if (h & kFlagBounds) return CLEF_ERR_DEVICE_BOUNDS;
    return CLEF_OK;
}

int clef_selftest_wait_timeout(void* workspace, int64_t limit_ns, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || limit_ns < 1000 || limit_ns > 100000000)
        return CLEF_ERR_INVALID_ARGUMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CK(cudaMemsetAsync(workspace, 0, 256, st));
    CK(launch_wait_timeout_selftest(static_cast<int*>(workspace), uint64_t(limit_ns), st));
    return CLEF_OK;
}

int clef_span_sums(const clef_config* cfg, const clef_schema* schema, const uint16_t* hidden,
                   const int32_t* token_ids, const uint16_t* lexical, float* q_sum, float* o_sum, float* x_sum,
                   void* workspace, size_t workspace_bytes, void* stream) {
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    if (!hidden || !token_ids || !lexical || !q_sum || !o_sum || !x_sum || !workspace) return CLEF_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(lexical) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(q_sum) & 15) ||
        (reinterpret_cast<uintptr_t>(o_sum) & 15) || (reinterpret_cast<uintptr_t>(x_sum) & 15))
        return CLEF_ERR_INVALID_ARGUMENT;
    const Plan* pp = nullptr;
    const WsLayout* lp = nullptr;
    const int v = cached_plan(cfg, schema, &pp, &lp);
    if (v != CLEF_OK) return v;
    const Plan& p = *pp;
    const WsLayout& L = *lp;
    if (workspace_bytes < L.total) return CLEF_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int u = upload_plan(p, ws, ws + L.plan, st);
    if (u != CLEF_OK) return u;
    const int32_t* plan = reinterpret_cast<const int32_t*>(ws + L.plan);
    SpanPoolArgs sp{};
    sp.hidden = hidden; sp.row_stride = schema->row_stride; sp.Lpad = schema->Lpad; sp.H = cfg->hidden;
    sp.vocab = cfg->vocab; sp.token_ids = token_ids; sp.lexical = lexical;
    sp.items = reinterpret_cast<const int4*>(plan + p.item);
    sp.lengths = plan + p.lengths; sp.rec_row_off = plan + p.rec_row_off; sp.rec_q_off = plan + p.rec_q_off;
    sp.q_rec = plan + p.q_rec; sp.q_span = plan + p.q_span; sp.q_opt_off = plan + p.q_opt_off;
    sp.o_rec = plan + p.o_rec; sp.o_span = plan + p.o_span;
    sp.q_sum = q_sum; sp.o_sum = o_sum; sp.x_sum = x_sum;
    sp.flags = reinterpret_cast<int*>(ws + L.flags);
    CK(launch_span_pool(sp, p.n_items, true, st));
    return CLEF_OK;
}

uint64_t clef_kernel_launches(void) { return g_kernel_launches.load(); }

int clef_gemm_bf16(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, const float* bias, float* C,
                   int64_t ldc, int32_t M, int32_t N, int32_t K, int32_t* flags, void* stream) {
    if (!A || !B || !C || !flags) return CLEF_ERR_INVALID_ARGUMENT;
    if (M < 1 || N < 1 || K < 1 || K % 64 || N % 64 || lda % 8 || ldb % 8 || lda < K || ldb < K || ldc < N ||
        ldc % 4)
        return CLEF_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (reinterpret_cast<uintptr_t>(C) & 15))
        return CLEF_ERR_INVALID_ARGUMENT;
    GemmProblem g;
    g.A = A; g.lda = lda; g.a_rows = M; g.B = B; g.ldb = ldb; g.N = N; g.K = K;
    g.n_mtiles = (M + kTile - 1) / kTile;
    GemmEpilogue e;
    e.kind = EPI_F32; e.bias_f32 = bias; e.out = C; e.ldo = ldc; e.M = M;
    CK(launch_gemm(g, e, flags, static_cast<cudaStream_t>(stream)));
    return CLEF_OK;
}

// ------------------------------------------------ allocation-free span sums

}  // extern "C"

// Scratch of clef_span_sums_noalloc: the status word (first 256 bytes) and the plan.
// On the host this name is only a stand-in, not a device address: host code looks
// the device address up once per device and passes that to the kernel.
static __device__ __align__(256) uint8_t g_span_sums_scratch[CLEF_SPAN_SUMS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up on first use).
int span_sums_scratch(uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CLEF_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_span_sums_scratch) != cudaSuccess || !p) return CLEF_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
    return CLEF_OK;
}

}  // namespace

extern "C" {

int clef_span_sums_noalloc(const clef_config* cfg, const clef_schema* schema, const uint16_t* hidden,
                           const int32_t* token_ids, const uint16_t* lexical, float* q_sum, float* o_sum,
                           float* x_sum, void* stream) {
    if (!config_ok(cfg)) return CLEF_ERR_UNSUPPORTED_CONFIG;
    if (!hidden || !token_ids || !lexical || !q_sum || !o_sum || !x_sum) return CLEF_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(lexical) & 15) ||
        (reinterpret_cast<uintptr_t>(q_sum) & 15) || (reinterpret_cast<uintptr_t>(o_sum) & 15) ||
        (reinterpret_cast<uintptr_t>(x_sum) & 15))
        return CLEF_ERR_INVALID_ARGUMENT;
    const Plan* pp = nullptr;
    const WsLayout* lp = nullptr;
    const int v = cached_plan(cfg, schema, &pp, &lp);
    if (v != CLEF_OK) return v;
    const Plan& p = *pp;
    constexpr size_t kPlanOff = 256;  // the status word sits in the first 256 bytes
    if (kPlanOff + p.blob.size() * 4 > CLEF_SPAN_SUMS_NOALLOC_SCRATCH_BYTES) return CLEF_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* scratch = nullptr;
    const int sa = span_sums_scratch(&scratch);
    if (sa != CLEF_OK) return sa;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    {
        const int u = upload_plan(p, scratch, scratch + kPlanOff, st);  // also clears the status word
        if (u != CLEF_OK) return u;
    }
    const int32_t* plan = reinterpret_cast<const int32_t*>(scratch + kPlanOff);
    SpanPoolArgs sp{};
    sp.hidden = hidden; sp.row_stride = schema->row_stride; sp.Lpad = schema->Lpad; sp.H = cfg->hidden;
    sp.vocab = cfg->vocab; sp.token_ids = token_ids; sp.lexical = lexical;
    sp.items = reinterpret_cast<const int4*>(plan + p.item);
    sp.lengths = plan + p.lengths; sp.rec_row_off = plan + p.rec_row_off; sp.rec_q_off = plan + p.rec_q_off;
    sp.q_rec = plan + p.q_rec; sp.q_span = plan + p.q_span; sp.q_opt_off = plan + p.q_opt_off;
    sp.o_rec = plan + p.o_rec; sp.o_span = plan + p.o_span;
    sp.q_sum = q_sum; sp.o_sum = o_sum; sp.x_sum = x_sum;
    sp.flags = reinterpret_cast<int*>(scratch);
    CK(launch_span_pool(sp, p.n_items, true, st));
    int h = 0;
    CK(cudaMemcpyAsync(&h, scratch, 4, cudaMemcpyDeviceToHost, st));
    CK(cudaStreamSynchronize(st));
    if (h & kFlagTimeout) return CLEF_ERR_DEVICE_TIMEOUT;
    if (h & kFlagBounds) return CLEF_ERR_DEVICE_BOUNDS;
    return CLEF_OK;
}

}  // extern "C"
