// The per-record tail of the JointSchemaHead in one launch: option LayerNorm, field
// aggregation ("clef-4bit JointSchemaHead walkthrough" section 3 step 3: question base
// vector + option-weighted summary + global vector + type embedding), the joint
// transformer layers over the record's fields (section 3 step 3; "Dissecting the
// Clef-Flash architecture" section 3.2: 4 layers, width 1024, 16 heads, feed-forward
// 4096), the field LayerNorm, and the scorer with the per-question softmax (section 3
// step 4; "clef-flash-CoreAI metadata.json" decision.softmax and decision.response).
//
// One thread-block cluster of 16 CTAs per group of consecutive records (at most 48
// fields and 256 options; the host packs records into about as many groups as the GPU
// holds clusters at once).  CTA r owns width columns [64 r, 64 r + 64) of every
// width-D activation -- attention head r -- and the matching rows of every weight
// matrix.  Those rows are prepared once as contiguous, pre-swizzled 64-column tiles
// (launch_tail_slices), so each pipeline stage brings its weight tiles in with one
// bulk copy and its activation rows with TMA, through an mbarrier ring fed by a
// producer warp, into mma.sync bf16 tensor-core tiles whose M is the group's fields or
// options (16-row tiles, as many as the rows need).  Activations whose whole rows every CTA needs (LayerNorm outputs, the
// attention output, the feed-forward hidden layer, the scorer input) go through L2 in
// the workspace, with a cluster barrier between writer and readers.  LayerNorm
// statistics combine each CTA's (mean, M2) pair per row through distributed shared
// memory.  The field self-attention of head r is local to CTA r (fields attend only to
// fields of their own record).  Every reduction runs
// in a fixed order, so results do not depend on timing.  No CTA waits on a flag: the
// cluster barrier is a hardware barrier every thread passes on every path.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "head_kernels.h"
#include "kernels.h"

namespace clef {

namespace {

constexpr int CL = 16;                     // CTAs per record
constexpr int kW = 1024;                   // width the kernel is built for
constexpr int kCols = kW / CL;             // width columns (one head) per CTA
constexpr int kFF = 4096;                  // feed-forward width the kernel is built for
constexpr int kConsumers = 8;              // MMA warps
constexpr int kThreads = (kConsumers + 1) * 32;  // + 1 TMA producer warp (it joins the non-GEMM phases)
constexpr int kKC = 64;                    // K per pipeline stage (one 128-byte swizzled row per operand row)
constexpr int kStages = 5;                 // stages of the largest tiles (FFN hidden projection)
constexpr int kMaxStages = 16;             // stages of smaller tiles: as many as fit kPipeBytes
constexpr int kMaxQ = kMaxFields;          // 48 fields: 3 m16 tiles
constexpr int kBoxF = kMaxQ;               // A rows loaded per stage for the field projections
constexpr int kBoxO = 128;                 // A rows loaded per stage for the scorer MLP (8 m16 tiles)
constexpr int kMaxO = kTailMaxRecOptions;  // 256
constexpr int kStageBytes = (kBoxF + 256) * 128 > (kBoxO + 64) * 128 ? (kBoxF + 256) * 128 : (kBoxO + 64) * 128;
constexpr int kPipeBytes = kStages * kStageBytes;
constexpr int kQkvLd = 3 * kCols + 1;      // attention scratch row stride (floats)
static_assert(kStageBytes % 1024 == 0 && (kBoxF * 128) % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
static_assert(kMaxO * kCols * 4 <= kPipeBytes, "option slice staging fits the pipeline buffers");
static_assert((kMaxQ * kQkvLd + kMaxQ * (kMaxQ + 1)) * 4 <= kPipeBytes, "attention scratch fits the pipeline buffers");
static_assert(kMaxO <= kThreads, "one thread per option in the pooling scores");
static_assert(32 * kBoxO * 4 <= kPipeBytes, "MLP partials per (warp, quad lane) fit the pipeline buffers");

// Tensor maps of the activation operands (bf16, 64-element x box_rows boxes, 128-byte swizzle).
enum TailMap { kMapAField = 0, kMapLn, kMapAttn, kMapHid, kMapZ, kNumMaps };

// Shared memory of one CTA (offsets from the 1024-byte aligned base).
constexpr int kOffPipe = 0;
constexpr int kOffF = kOffPipe + kPipeBytes;           // float [kMaxQ][kCols]: f, then f_hat (this CTA's columns)
constexpr int kOffPart = kOffF + kMaxQ * kCols * 4;    // float [kMaxO][2]: LayerNorm (mean, M2) partials (cluster-read)
constexpr int kOffStat = kOffPart + kMaxO * 2 * 4;     // float [kMaxO][2]: row mean, rstd
constexpr int kOffDot = kOffStat + kMaxO * 2 * 4;      // float [kMaxO]: pooling-score partials (cluster-read)
constexpr int kOffAlpha = kOffDot + kMaxO * 4;         // float [kMaxO]: option pooling weights / scores
constexpr int kOffSPart = kOffAlpha + kMaxO * 4;       // float [kMaxO][5]: scorer partials (cluster-read)
constexpr int kOffQPart = kOffSPart + kMaxO * 5 * 4;   // float [kMaxQ][2]: scorer per-question partials (cluster-read)
constexpr int kOffBar = kOffQPart + kMaxQ * 2 * 4;     // uint64 [2][kMaxStages]: stage full / empty barriers
constexpr int kSmemBytes = kOffBar + 2 * kMaxStages * 8 + 1024;
static_assert(kSmemBytes <= 232448, "fits one CTA's shared memory");

__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(saddr));
}
// Plain loads of another CTA's shared memory (cluster addresses from cluster_map); the
// callers order them with cluster_sync().  Volatile, so that they stay after that
// barrier; callers issue all loads of a reduction before summing, so they overlap.
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// byte offset of 16-byte chunk `chunk` of row `row` in a tile written by TMA with the
// 128-byte swizzle (tile base 1024-byte aligned)
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// The stage ring.  Each GEMM streams its K range in chunks of NB boxes of 64 columns
// through as many stages of its own size as the pipeline buffers hold (at most
// kMaxStages), from stage 0 (every stage is free when a GEMM starts).  Warp kConsumers
// (lane 0) is the producer: it waits for a stage's `empty` barrier (one arrival per
// consumer warp) and refills it with TMA, so the consumer warps never synchronise with
// each other inside a GEMM.  Every thread of a role runs the same GEMMs, so the parity
// bits below are the same in every thread of the role.
struct Ring {
    uint64_t* full;     // [kMaxStages], completed by the TMA bytes
    uint64_t* empty;    // [kMaxStages], kConsumers arrivals
    uint32_t fp;        // consumers: bit s = parity of full[s]'s next completion
    uint32_t ep;        // producer: bit s = parity of empty[s]'s next completion
    uint32_t used;      // producer: bit s = stage s has been filled before
    volatile int* failed;
    int* flags;
};

// One bulk copy of `bytes` contiguous bytes into this CTA's shared memory, completing
// on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// C[m][n] = sum_k A[m][k] B[n][k] over nk chunks of NB * 64 columns, for m < 16 MT and
// n < 64 NT8 (consumer warp w owns columns [8 NT8 w, 8 NT8 (w + 1))).  A stage holds the
// NB A boxes (a_bytes each) followed by the NB B tiles (b_bytes each, 64 NT8 rows).
// issue(kc, stage, bar) -- producer thread only -- starts the copies of chunk kc into
// `stage` (the barrier is armed for NB (a_bytes + b_bytes) bytes before).
// epi(row, col, v0, v1) gets columns col, col + 1 of every row < m_rows (consumer warps).
template <int MT, int NT8, int NB, typename Issue, typename Epi>
__device__ __forceinline__ void tile_gemm(Ring& ring, uint8_t* pipe, int nk, int a_bytes, int b_bytes, int m_rows,
                                          Issue issue, Epi epi) {
    const int stage_bytes = NB * (a_bytes + b_bytes);
    const int S = min(kMaxStages, kPipeBytes / stage_bytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kConsumers) {
        if (lane == 0) {
            fence_proxy_async_global();  // A rows written by generic stores are read by TMA
            int st = 0;
            for (int kc = 0; kc < nk; ++kc) {
                if ((ring.used >> st) & 1u) {
                    if (!*ring.failed &&
                        !mbar_wait_bounded(&ring.empty[st], (ring.ep >> st) & 1u, ring.failed, ring.flags))
                        *ring.failed = 1;
                    ring.ep ^= 1u << st;
                }
                ring.used |= 1u << st;
                mbar_arrive_expect_tx(&ring.full[st], uint32_t(stage_bytes));
                issue(kc, pipe + st * stage_bytes, &ring.full[st]);
                if (++st == S) st = 0;
            }
        }
        __syncwarp();
    } else {
        float acc[MT][NT8][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
        int st = 0;
        for (int kc = 0; kc < nk; ++kc) {
            if (!*ring.failed && !mbar_wait_bounded(&ring.full[st], (ring.fp >> st) & 1u, ring.failed, ring.flags))
                *ring.failed = 1;
            ring.fp ^= 1u << st;
            const uint32_t s0 = smem_u32(pipe + st * stage_bytes);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint32_t a0 = s0 + uint32_t(b * a_bytes), b0 = s0 + uint32_t(NB * a_bytes + b * b_bytes);
#pragma unroll
                for (int ks = 0; ks < kKC / 16; ++ks) {
                    uint32_t af[MT][4];
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        ldmatrix_x4(af[mt], a0 + swz(mt * 16 + (lane & 15), ks * 2 + (lane >> 4)));
#pragma unroll
                    for (int nt = 0; nt < NT8; ++nt) {
                        uint32_t bf[2];
                        const int n = warp * 8 * NT8 + nt * 8 + (lane & 7);
                        ldmatrix_x2(bf, b0 + swz(n, ks * 2 + ((lane >> 3) & 1)));
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(acc[mt][nt], af[mt], bf[0], bf[1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.empty[st]);  // this warp is done with the stage
            if (++st == S) st = 0;
        }
        const int g = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = mt * 16 + g + 8 * h;
                    if (row < m_rows)
                        epi(row, warp * 8 * NT8 + nt * 8 + 2 * tq, acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]);
                }
    }
    __syncthreads();  // every stage is consumed and the epilogue is done
}

// A projection of the group's fields: as many 16-row tiles as the fields need; the A
// rows come from activation map `amap` at row q0, the B tiles (64 NT8 rows of this CTA,
// NB per chunk) from the sliced weights at `wslice`.
template <int NT8, int NB, typename Epi>
__device__ __forceinline__ void field_gemm(Ring& ring, uint8_t* pipe, int K, int m_rows, const CUtensorMap* amap,
                                           int q0, const uint16_t* wslice, Epi epi) {
    constexpr int a_bytes = kBoxF * 128, b_bytes = 64 * NT8 * 128;
    static_assert(NB * (a_bytes + b_bytes) <= kPipeBytes / 2, "at least two stages");
    const int nk = K / (kKC * NB);
    auto issue = [&](int kc, uint8_t* st, uint64_t* bar) {
#pragma unroll
        for (int b = 0; b < NB; ++b) tma_load_2d(st + b * a_bytes, amap, (kc * NB + b) * kKC, q0, bar);
        bulk_load(st + NB * a_bytes, reinterpret_cast<const uint8_t*>(wslice) + int64_t(kc) * NB * b_bytes,
                  uint32_t(NB * b_bytes), bar);
    };
    if (m_rows <= 16) tile_gemm<1, NT8, NB>(ring, pipe, nk, a_bytes, b_bytes, m_rows, issue, epi);
    else if (m_rows <= 32) tile_gemm<2, NT8, NB>(ring, pipe, nk, a_bytes, b_bytes, m_rows, issue, epi);
    else tile_gemm<3, NT8, NB>(ring, pipe, nk, a_bytes, b_bytes, m_rows, issue, epi);
}

// First element of CTA r's tiles in a sliced weight matrix of K columns, R rows per CTA.
__device__ __forceinline__ const uint16_t* slice_of(const uint16_t* w, int r, int R, int K) {
    return w + int64_t(r) * R * K;
}

// Row mean and 1/sqrt(var + eps) over the full width of n rows, this CTA holding
// columns [64 r, 64 r + 64) of them in x (row stride ldx floats): each CTA's (mean, M2)
// per row goes to `part`, and after a cluster barrier every CTA combines the 16 pairs
// in rank order (parallel-variance merge of equal-size parts).  The caller keeps `part`
// untouched until the next cluster barrier after this call.
__device__ void cluster_row_stats(const float* x, int ldx, int n, float* part, float* stat) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < n; i += kThreads / 32) {
        const float v0 = x[i * ldx + lane], v1 = x[i * ldx + lane + 32];
        const float m = warp_sum(v0 + v1) * (1.0f / kCols);
        const float m2 = warp_sum((v0 - m) * (v0 - m) + (v1 - m) * (v1 - m));
        if (lane == 0) {
            part[2 * i] = m;
            part[2 * i + 1] = m2;
        }
    }
    cluster_sync();
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t p = smem_u32(part + 2 * i);
        float2 v[CL];
#pragma unroll
        for (int r = 0; r < CL; ++r) v[r] = ld_cluster_f2(cluster_map(p, uint32_t(r)));
        float msum = 0.f, m2 = 0.f;
#pragma unroll
        for (int r = 0; r < CL; ++r) {
            msum += v[r].x;
            m2 += v[r].y;
        }
        const float mu = msum * (1.0f / CL);
#pragma unroll
        for (int r = 0; r < CL; ++r) m2 += float(kCols) * (v[r].x - mu) * (v[r].x - mu);
        stat[2 * i] = mu;
        stat[2 * i + 1] = rsqrtf(m2 * (1.0f / kW) + 1e-5f);
    }
    __syncthreads();
}

// LayerNorm of this CTA's columns of n rows (x, row stride kCols) written as bf16 into
// columns [64 r, 64 r + 64) of rows of a global [*, kW] matrix.
__device__ void ln_write_bf16(const float* x, int n, const float* stat, const uint16_t* w, const uint16_t* b, int r,
                              uint16_t* out) {
    for (int i = threadIdx.x; i < n * (kCols / 2); i += kThreads) {
        const int row = i / (kCols / 2), c = (i % (kCols / 2)) * 2;
        const float mu = stat[2 * row], rs = stat[2 * row + 1];
        const int col = r * kCols + c;
        const float y0 = (x[row * kCols + c] - mu) * rs * bf16_to_float(w[col]) + bf16_to_float(b[col]);
        const float y1 = (x[row * kCols + c + 1] - mu) * rs * bf16_to_float(w[col + 1]) + bf16_to_float(b[col + 1]);
        *reinterpret_cast<uint32_t*>(out + int64_t(row) * kW + col) = pack_bf16(y0, y1);
    }
}

}  // namespace

struct TailMaps {
    CUtensorMap m[kNumMaps];
};

__global__ void __launch_bounds__(kThreads, 1)
    record_tail_kernel(const __grid_constant__ TailMaps maps, const RecordTailArgs a) {
    griddep_wait();
    griddep_launch();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* pipe = smem + kOffPipe;
    float* fs = reinterpret_cast<float*>(smem + kOffF);
    float* part = reinterpret_cast<float*>(smem + kOffPart);
    float* stat = reinterpret_cast<float*>(smem + kOffStat);
    float* dpart = reinterpret_cast<float*>(smem + kOffDot);
    float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
    float* spart = reinterpret_cast<float*>(smem + kOffSPart);
    float* qpart = reinterpret_cast<float*>(smem + kOffQPart);
    float* mw = reinterpret_cast<float*>(pipe);  // [32][kBoxO] after each scorer GEMM
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* empty = full + kMaxStages;
    __shared__ int failed;

    const int r = int(cluster_ctarank());
    const int grp = int(blockIdx.x) / CL;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tq = lane & 3;
    const int H = a.H;
    const int rb0 = a.grp_rec[grp], rb1 = a.grp_rec[grp + 1];
    const int q0 = a.rec_q_off[rb0], nq = a.rec_q_off[rb1] - q0;
    const int o0 = a.rec_o_off[rb0], no = a.rec_o_off[rb1] - o0;
    const int c0 = r * kCols;  // this CTA's first width column

    if (threadIdx.x == 0) {
        for (int st = 0; st < kMaxStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kConsumers);
        }
        failed = 0;
        fence_barrier_init();
        for (int m = 0; m < kNumMaps; ++m) prefetch_tensormap(&maps.m[m]);
    }
    __syncthreads();
    Ring ring{full, empty, 0u, 0u, 0u, &failed, a.flags};

    // ---------------------------------------------- option LayerNorm, pooling scores
    {
        float* ohs = reinterpret_cast<float*>(pipe);  // [no][kCols]: o, then o_hat (this CTA's columns)
        for (int i = threadIdx.x; i < no * (kCols / 4); i += kThreads) {
            const int j = i / (kCols / 4), c = (i % (kCols / 4)) * 4;
            *reinterpret_cast<float4*>(ohs + j * kCols + c) =
                *reinterpret_cast<const float4*>(a.o_res + int64_t(o0 + j) * kW + c0 + c);
        }
        __syncthreads();
        cluster_row_stats(ohs, kCols, no, part, stat);
        const float wa0 = bf16_to_float(a.pool_w[c0 + lane]), wa1 = bf16_to_float(a.pool_w[c0 + lane + 32]);
        const float g0 = bf16_to_float(a.opt_ln_w[c0 + lane]), g1 = bf16_to_float(a.opt_ln_w[c0 + lane + 32]);
        const float e0 = bf16_to_float(a.opt_ln_b[c0 + lane]), e1 = bf16_to_float(a.opt_ln_b[c0 + lane + 32]);
        for (int j = warp; j < no; j += kThreads / 32) {
            const float mu = stat[2 * j], rs = stat[2 * j + 1];
            const float y0 = (ohs[j * kCols + lane] - mu) * rs * g0 + e0;
            const float y1 = (ohs[j * kCols + lane + 32] - mu) * rs * g1 + e1;
            ohs[j * kCols + lane] = y0;
            ohs[j * kCols + lane + 32] = y1;
            a.o_hat[int64_t(o0 + j) * kW + c0 + lane] = y0;
            a.o_hat[int64_t(o0 + j) * kW + c0 + lane + 32] = y1;
            const float d = warp_sum(y0 * wa0 + y1 * wa1);
            if (lane == 0) dpart[j] = d;
        }
        cluster_sync();  // every CTA's pooling-score partials are complete
        // pooling score of every option of the group (each CTA computes all of them)
        if (threadIdx.x < no) {
            const uint32_t p = smem_u32(dpart + threadIdx.x);
            float d[CL];
#pragma unroll
            for (int rr = 0; rr < CL; ++rr) d[rr] = ld_cluster_f32(cluster_map(p, uint32_t(rr)));
            float sc = bf16_to_float(a.pool_b[0]);
#pragma unroll
            for (int rr = 0; rr < CL; ++rr) sc += d[rr];
            alpha[threadIdx.x] = sc;
        }
        __syncthreads();
        // alpha = softmax of the scores over each question's options
        for (int k = warp; k < nq; k += kThreads / 32) {
            const int j0 = a.q_opt_off[q0 + k] - o0, n = a.q_opt_off[q0 + k + 1] - o0 - j0;
            float m = -INFINITY;
            for (int j = lane; j < n; j += 32) m = fmaxf(m, alpha[j0 + j]);
            m = warp_max(m);
            float zs = 0.f;
            for (int j = lane; j < n; j += 32) zs += expf(alpha[j0 + j] - m);
            zs = warp_sum(zs);
            __syncwarp();
            for (int j = lane; j < n; j += 32) alpha[j0 + j] = expf(alpha[j0 + j] - m) / zs;
        }
        __syncthreads();
        // option-weighted summary of this CTA's columns, written as bf16 into the field
        // projection's input row
        for (int i = threadIdx.x; i < nq * (kCols / 2); i += kThreads) {
            const int k = i / (kCols / 2), c = (i % (kCols / 2)) * 2;
            const int j0 = a.q_opt_off[q0 + k] - o0, j1 = a.q_opt_off[q0 + k + 1] - o0;
            float s0 = 0.f, s1 = 0.f;
            for (int j = j0; j < j1; ++j) {
                s0 += alpha[j] * ohs[j * kCols + c];
                s1 += alpha[j] * ohs[j * kCols + c + 1];
            }
            *reinterpret_cast<uint32_t*>(a.a_field + int64_t(q0 + k) * a.ld_field + 2 * H + c0 + c) =
                pack_bf16(s0, s1);
        }
        fence_proxy_async_global();
        cluster_sync();  // every CTA's summary columns are in L2; the score partials are read
    }

    // ------------------------------------------------------------- field projection
    {
        const int K = 2 * H + kW;
        field_gemm<1, 4>(ring, pipe, K, nq, &maps.m[kMapAField], q0, slice_of(a.w_field, r, kCols, K),
                      [&](int row, int col, float v0, float v1) {
                          const int t = a.q_type[q0 + row] * kW + c0 + col;
                          fs[row * kCols + col] = v0 + bf16_to_float(a.b_field[c0 + col]) + bf16_to_float(a.type_emb[t]);
                          fs[row * kCols + col + 1] =
                              v1 + bf16_to_float(a.b_field[c0 + col + 1]) + bf16_to_float(a.type_emb[t + 1]);
                      });
        __syncthreads();
    }

    // --------------------------------------------------------------- joint layers
    for (int li = 0; li < a.n_joint; ++li) {
        // pre-attention LayerNorm -> ln_buf
        cluster_row_stats(fs, kCols, nq, part, stat);
        ln_write_bf16(fs, nq, stat, a.ln1_w[li], a.ln1_b[li], r, a.ln_buf + int64_t(q0) * kW);
        fence_proxy_async_global();
        cluster_sync();
        // q, k, v of head r
        float* qkv = reinterpret_cast<float*>(pipe);  // used after the GEMM
        field_gemm<3, 2>(ring, pipe, kW, nq, &maps.m[kMapLn], q0, slice_of(a.w_qkv[li], r, 3 * kCols, kW),
                      [&](int row, int col, float v0, float v1) {
                          const uint16_t* bq = a.b_qkv[li] + (col / kCols) * kW + c0 + col % kCols;
                          qkv[row * kQkvLd + col] = v0 + bf16_to_float(bq[0]);
                          qkv[row * kQkvLd + col + 1] = v1 + bf16_to_float(bq[1]);
                      });
        __syncthreads();
        // self-attention of head r among the fields of each record (all mutually visible)
        {
            float* sc = qkv + kMaxQ * kQkvLd;  // [kMaxQ][kMaxQ + 1]
            for (int i = threadIdx.x; i < nq * nq; i += kThreads) {
                const int x = i / nq, y = i % nq;
                float s = -INFINITY;
                if (a.q_rec[q0 + x] == a.q_rec[q0 + y]) {
                    const float* qx = qkv + x * kQkvLd;
                    const float* ky = qkv + y * kQkvLd + kCols;
                    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int d = 0; d < kCols; d += 4) {
                        s4[0] += qx[d] * ky[d];
                        s4[1] += qx[d + 1] * ky[d + 1];
                        s4[2] += qx[d + 2] * ky[d + 2];
                        s4[3] += qx[d + 3] * ky[d + 3];
                    }
                    s = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * 0.125f;  // 1 / sqrt(64)
                }
                sc[x * (kMaxQ + 1) + y] = s;
            }
            __syncthreads();
            for (int x = warp; x < nq; x += kThreads / 32) {
                float m = -INFINITY;
                for (int y = lane; y < nq; y += 32) m = fmaxf(m, sc[x * (kMaxQ + 1) + y]);
                m = warp_max(m);
                float zs = 0.f;
                for (int y = lane; y < nq; y += 32) zs += expf(sc[x * (kMaxQ + 1) + y] - m);
                zs = warp_sum(zs);
                __syncwarp();
                for (int y = lane; y < nq; y += 32) sc[x * (kMaxQ + 1) + y] = expf(sc[x * (kMaxQ + 1) + y] - m) / zs;
            }
            __syncthreads();
            for (int i = threadIdx.x; i < nq * (kCols / 2); i += kThreads) {
                const int x = i / (kCols / 2), d = (i % (kCols / 2)) * 2;
                float o0v = 0.f, o1v = 0.f;
                for (int y = 0; y < nq; ++y) {
                    const float pv = sc[x * (kMaxQ + 1) + y];
                    o0v += pv * qkv[y * kQkvLd + 2 * kCols + d];
                    o1v += pv * qkv[y * kQkvLd + 2 * kCols + d + 1];
                }
                *reinterpret_cast<uint32_t*>(a.attn_buf + int64_t(q0 + x) * kW + c0 + d) = pack_bf16(o0v, o1v);
            }
        }
        fence_proxy_async_global();
        cluster_sync();
        // output projection, residual
        field_gemm<1, 4>(ring, pipe, kW, nq, &maps.m[kMapAttn], q0, slice_of(a.w_o[li], r, kCols, kW),
                      [&](int row, int col, float v0, float v1) {
                          fs[row * kCols + col] += v0 + bf16_to_float(a.b_o[li][c0 + col]);
                          fs[row * kCols + col + 1] += v1 + bf16_to_float(a.b_o[li][c0 + col + 1]);
                      });
        __syncthreads();
        // pre-FFN LayerNorm -> ln_buf
        cluster_row_stats(fs, kCols, nq, part, stat);
        ln_write_bf16(fs, nq, stat, a.ln2_w[li], a.ln2_b[li], r, a.ln_buf + int64_t(q0) * kW);
        fence_proxy_async_global();
        cluster_sync();
        // FFN hidden columns [256 r, 256 r + 256), GELU -> hid_buf
        {
            constexpr int kHc = kFF / CL;
            field_gemm<4, 1>(ring, pipe, kW, nq, &maps.m[kMapLn], q0, slice_of(a.w_1[li], r, kHc, kW),
                          [&](int row, int col, float v0, float v1) {
                              const int hc = r * kHc + col;
                              const float h0 = gelu_exact(v0 + bf16_to_float(a.b_1[li][hc]));
                              const float h1 = gelu_exact(v1 + bf16_to_float(a.b_1[li][hc + 1]));
                              *reinterpret_cast<uint32_t*>(a.hid_buf + int64_t(q0 + row) * kFF + hc) = pack_bf16(h0, h1);
                          });
        }
        fence_proxy_async_global();
        cluster_sync();
        // FFN output projection, residual
        field_gemm<1, 4>(ring, pipe, kFF, nq, &maps.m[kMapHid], q0, slice_of(a.w_2[li], r, kCols, kFF),
                      [&](int row, int col, float v0, float v1) {
                          fs[row * kCols + col] += v0 + bf16_to_float(a.b_2[li][c0 + col]);
                          fs[row * kCols + col + 1] += v1 + bf16_to_float(a.b_2[li][c0 + col + 1]);
                      });
        __syncthreads();
    }

    // --------------------------------------------------- field LayerNorm -> f_hat
    cluster_row_stats(fs, kCols, nq, part, stat);
    for (int i = threadIdx.x; i < nq * kCols; i += kThreads) {
        const int row = i / kCols, c = i % kCols;
        const float y = (fs[i] - stat[2 * row]) * stat[2 * row + 1] * bf16_to_float(a.fld_ln_w[c0 + c]) +
                        bf16_to_float(a.fld_ln_b[c0 + c]);
        fs[i] = y;
        a.f_hat[int64_t(q0 + row) * kW + c0 + c] = y;
    }
    __syncthreads();

    // ------------------------------------------------------------------- scorer
    // scorer input z_j = [f_hat_q, o_hat_j, f_hat_q * o_hat_j, |f_hat_q - o_hat_j|] (this
    // CTA's columns of each segment), and the partial sums of the joint cosine
    for (int j = warp; j < no; j += kThreads / 32) {
        const int k = a.o_q[o0 + j] - q0;
        float fo = 0.f, oo = 0.f;
        uint16_t* zr = a.z + int64_t(o0 + j) * 4 * kW + c0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = lane + 32 * h;
            const float f = fs[k * kCols + c], o = a.o_hat[int64_t(o0 + j) * kW + c0 + c];
            zr[c] = float_to_bf16(f);
            zr[kW + c] = float_to_bf16(o);
            zr[2 * kW + c] = float_to_bf16(f * o);
            zr[3 * kW + c] = float_to_bf16(fabsf(f - o));
            fo += f * o;
            oo += o * o;
        }
        fo = warp_sum(fo);
        oo = warp_sum(oo);
        if (lane == 0) {
            spart[j * 5 + 1] = fo;
            spart[j * 5 + 2] = oo;
        }
    }
    // prior partials over this CTA's share of the backbone width: x . (u + g), |x|^2, |u + g|^2
    {
        const int hc = H / CL, h0 = r * hc;  // hc = 256 or 320: 8 or 10 float4 groups of 32 lanes / 4
        constexpr int kMaxV = 3;             // float4 loads per lane per option (hc <= 384)
        for (int j = warp; j < no; j += kThreads / 32) {
            const int q = a.o_q[o0 + j];
            const float4* gv = reinterpret_cast<const float4*>(a.g32 + int64_t(a.q_rec[q]) * H + h0);
            const float4* xv = reinterpret_cast<const float4*>(a.x32 + int64_t(o0 + j) * H + h0);
            const float4* uv = reinterpret_cast<const float4*>(a.u32 + int64_t(q) * H + h0);
            float4 x4[kMaxV], u4[kMaxV], g4[kMaxV];
#pragma unroll
            for (int v = 0; v < kMaxV; ++v) {  // every load of the option in flight at once
                const int c = lane + 32 * v;
                if (c < hc / 4) {
                    x4[v] = xv[c];
                    u4[v] = uv[c];
                    g4[v] = gv[c];
                }
            }
            float xa = 0.f, xx = 0.f;
#pragma unroll
            for (int v = 0; v < kMaxV; ++v) {
                if (lane + 32 * v < hc / 4) {
                    xa += x4[v].x * (u4[v].x + g4[v].x) + x4[v].y * (u4[v].y + g4[v].y) +
                          x4[v].z * (u4[v].z + g4[v].z) + x4[v].w * (u4[v].w + g4[v].w);
                    xx += x4[v].x * x4[v].x + x4[v].y * x4[v].y + x4[v].z * x4[v].z + x4[v].w * x4[v].w;
                }
            }
            xa = warp_sum(xa);
            xx = warp_sum(xx);
            if (lane == 0) {
                spart[j * 5 + 3] = xa;
                spart[j * 5 + 4] = xx;
            }
        }
        for (int k = warp; k < nq; k += kThreads / 32) {
            const float* gv = a.g32 + int64_t(a.q_rec[q0 + k]) * H + h0;
            const float* uv = a.u32 + int64_t(q0 + k) * H + h0;
            float aa = 0.f, ff = 0.f;
            for (int c = lane; c < hc; c += 32) {
                const float v = uv[c] + gv[c];
                aa += v * v;
            }
            for (int c = lane; c < kCols; c += 32) ff += fs[k * kCols + c] * fs[k * kCols + c];
            aa = warp_sum(aa);
            ff = warp_sum(ff);
            if (lane == 0) {
                qpart[2 * k] = ff;
                qpart[2 * k + 1] = aa;
            }
        }
    }
    fence_proxy_async_global();
    cluster_sync();  // every CTA's columns of z are in L2
    // scorer MLP hidden columns [64 r, 64 r + 64) and their share of w2 . GELU(.)
    for (int j0 = 0; j0 < no; j0 += kBoxO) {
        const int n = min(kBoxO, no - j0);
        constexpr int a_bytes = kBoxO * 128, b_bytes = 64 * 128, NB = 2;
        const uint8_t* wsl = reinterpret_cast<const uint8_t*>(slice_of(a.mlp1_w, r, kCols, 4 * kW));
        auto issue = [&](int kc, uint8_t* st, uint64_t* bar) {
#pragma unroll
            for (int b = 0; b < NB; ++b) tma_load_2d(st + b * a_bytes, &maps.m[kMapZ], (kc * NB + b) * kKC, o0 + j0, bar);
            bulk_load(st + NB * a_bytes, wsl + int64_t(kc) * NB * b_bytes, uint32_t(NB * b_bytes), bar);
        };
        auto epi = [&](int row, int col, float v0, float v1) {
            const float v = gelu_exact(v0 + bf16_to_float(a.mlp1_b[c0 + col])) * bf16_to_float(a.mlp2_w[c0 + col]) +
                            gelu_exact(v1 + bf16_to_float(a.mlp1_b[c0 + col + 1])) *
                                bf16_to_float(a.mlp2_w[c0 + col + 1]);
            mw[(warp * 4 + tq) * kBoxO + row] = v;
        };
        const int nk = 4 * kW / (kKC * NB);
        if (n <= 32) tile_gemm<2, 1, NB>(ring, pipe, nk, a_bytes, b_bytes, n, issue, epi);
        else if (n <= 64) tile_gemm<4, 1, NB>(ring, pipe, nk, a_bytes, b_bytes, n, issue, epi);
        else tile_gemm<8, 1, NB>(ring, pipe, nk, a_bytes, b_bytes, n, issue, epi);
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kThreads) {
            float sum = 0.f;
            for (int t = 0; t < 32; ++t) sum += mw[t * kBoxO + i];
            spart[(j0 + i) * 5] = sum;
        }
        __syncthreads();
    }
    cluster_sync();  // every CTA's scorer partials are complete
    // logits, softmax and answers of questions k = r, r + 16, ...: one warp per question
    {
        const float gate = 1.0f / (1.0f + expf(-bf16_to_float(a.gate[0])));
        const float jscale = bf16_to_float(a.joint_scale[0]);
        const float b2 = bf16_to_float(a.mlp2_b[0]);
        float* lg = alpha;  // reused: the logits of the questions this CTA finishes
        for (int k = r + CL * warp; k < nq; k += CL * (kThreads / 32)) {
            float2 qv[CL];
#pragma unroll
            for (int rr = 0; rr < CL; ++rr) qv[rr] = ld_cluster_f2(cluster_map(smem_u32(qpart + 2 * k), uint32_t(rr)));
            float ff = 0.f, aa = 0.f;
#pragma unroll
            for (int rr = 0; rr < CL; ++rr) {
                ff += qv[rr].x;
                aa += qv[rr].y;
            }
            const float nf = fmaxf(sqrtf(ff), 1e-8f), na = fmaxf(sqrtf(aa), 1e-8f);
            const int j0 = a.q_opt_off[q0 + k] - o0, j1 = a.q_opt_off[q0 + k + 1] - o0;
            for (int j = j0 + lane; j < j1; j += 32) {
                float t5[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
                const uint32_t pa = smem_u32(spart + j * 5);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // eight CTAs' partials in flight at a time
                    float pv[CL / 2][5];
#pragma unroll
                    for (int rr = 0; rr < CL / 2; ++rr) {
                        const uint32_t pr = cluster_map(pa, uint32_t(h * (CL / 2) + rr));
#pragma unroll
                        for (int t = 0; t < 5; ++t) pv[rr][t] = ld_cluster_f32(pr + 4u * t);
                    }
#pragma unroll
                    for (int rr = 0; rr < CL / 2; ++rr)
#pragma unroll
                        for (int t = 0; t < 5; ++t) t5[t] += pv[rr][t];
                }
                const float prior = t5[3] / (fmaxf(sqrtf(t5[4]), 1e-8f) * na);
                const float joint = t5[1] / (nf * fmaxf(sqrtf(t5[2]), 1e-8f));
                lg[j] = prior + gate * (jscale * joint + t5[0] + b2);
            }
            __syncwarp();
            const int n = j1 - j0;
            float m = -INFINITY;
            for (int j = lane; j < n; j += 32) m = fmaxf(m, lg[j0 + j]);
            m = warp_max(m);
            float zs = 0.f;
            for (int j = lane; j < n; j += 32) zs += expf(lg[j0 + j] - m);
            zs = warp_sum(zs);
            float ev = 0.f;
            for (int j = lane; j < n; j += 32) {
                const float pj = expf(lg[j0 + j] - m) / zs;
                a.logits[o0 + j0 + j] = lg[j0 + j];
                a.probs[o0 + j0 + j] = pj;
                ev += float(j) * pj;
            }
            ev = warp_sum(ev);
            if (lane == 0) {
                int kk = 0;  // first maximum in option order
                for (int j = 1; j < n; ++j)
                    if (lg[j0 + j] > lg[j0 + kk]) kk = j;
                const float pk = expf(lg[j0 + kk] - m) / zs;
                const int t = a.q_type[q0 + k];
                a.q_argmax[q0 + k] = kk;
                a.q_conf[q0 + k] = pk;
                a.q_value[q0 + k] = t == 0 ? expf(lg[j0] - m) / zs : (t == 1 ? pk : ev);
            }
        }
    }
    cluster_sync();  // no CTA leaves while another may still read its shared memory
}

int record_tail_clusters() {
    static std::once_flag once;
    static int n = 0;
    std::call_once(once, [] {
        if (cudaFuncSetAttribute(record_tail_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
            cudaFuncSetAttribute(record_tail_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                cudaSuccess) {
            cudaGetLastError();
            return;
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(CL);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, record_tail_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    });
    return n;
}

cudaError_t launch_record_tail(const RecordTailArgs& a, cudaStream_t s) {
    if (a.n_groups <= 0) return cudaSuccess;
    if (a.D != kW || a.F != kFF || a.n_joint > kTailMaxJoint || a.H % (64 * CL) != 0 || a.H > 6144)
        return cudaErrorInvalidValue;
    if (record_tail_clusters() <= 0) return cudaErrorNotSupported;
    TailMaps maps;
    const uint64_t H = uint64_t(a.H);
    bool ok = make_tma_2d_bf16(&maps.m[kMapAField], a.a_field, 2 * H + kW, uint64_t(a.Q), uint64_t(a.ld_field), kBoxF);
    ok = ok && make_tma_2d_bf16(&maps.m[kMapLn], a.ln_buf, kW, uint64_t(a.Q), kW, kBoxF);
    ok = ok && make_tma_2d_bf16(&maps.m[kMapAttn], a.attn_buf, kW, uint64_t(a.Q), kW, kBoxF);
    ok = ok && make_tma_2d_bf16(&maps.m[kMapHid], a.hid_buf, kFF, uint64_t(a.Q), kFF, kBoxF);
    ok = ok && make_tma_2d_bf16(&maps.m[kMapZ], a.z, 4 * kW, uint64_t(a.O), 4 * kW, kBoxO);
    if (!ok) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.n_groups * CL));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return counted(cudaLaunchKernelEx(&cfg, record_tail_kernel, maps, a));
}

bool record_tail_shape(int H, int D, int heads, int F, int n_joint) {
    return D == kW && heads == CL && F == kFF && n_joint <= kTailMaxJoint && H % (64 * CL) == 0 && H <= 6144;
}

__global__ void __launch_bounds__(256) tail_slices_kernel(const uint16_t* __restrict__ w, int K, int R, int qkv, int D,
                                                         uint16_t* __restrict__ dst) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;  // one 16-byte chunk of one tile row
    const int nkc = K / kKC;
    if (i >= int64_t(CL) * nkc * R * 8) return;
    const int c = int(i % 8);
    int64_t t = i / 8;
    const int j = int(t % R);
    t /= R;
    const int kc = int(t % nkc), r = int(t / nkc);
    const int64_t row = qkv ? int64_t(j / kCols) * D + int64_t(r) * kCols + j % kCols : int64_t(r) * R + j;
    const uint4 v = *reinterpret_cast<const uint4*>(w + row * K + int64_t(kc) * kKC + c * 8);
    uint8_t* tile = reinterpret_cast<uint8_t*>(dst) + ((int64_t(r) * nkc + kc) * R) * 128;
    *reinterpret_cast<uint4*>(tile + swz(j, c)) = v;
}

cudaError_t launch_tail_slices(const uint16_t* w, int K, int R, int qkv, int D, uint16_t* dst, cudaStream_t s) {
    const int64_t n = int64_t(CL) * (K / kKC) * R * 8;
    tail_slices_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(w, K, R, qkv, D, dst);
    return counted(cudaGetLastError());
}

}  // namespace clef
