// Dense bf16 contraction on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, used for every projection of the head:
//   - the memory K/V projection of both routing layers in one N = 4 * width GEMM,
//     with the memory LayerNorm folded into the epilogue ("clef-4bit JointSchemaHead
//     walkthrough" section 3 step 2: options attend the whole memory);
//   - the option-query, routing, field, joint-layer and scorer projections.
//
// Design: persistent CTAs (one per SM) walk 128 x BN output tiles.  Warp 0 is the
// TMA producer, warp 1 owns TMEM and issues tcgen05.mma (one thread), warps 2..5
// drain the fp32 accumulators from TMEM and run the epilogue.  Two TMEM
// accumulators let the epilogue of one tile overlap the mainloop of the next.
// Operand tiles are 64-element K slices with the 128-byte swizzle, two per pipeline
// stage except for single-CTA 256-wide tiles: the one MMA-issuing thread is the
// kernel's critical path, and a stage then costs it one wait, fence and commit pair per
// eight MMAs.  Tiles are visited N-fastest so that CTAs working at the same time share
// A tiles in L2.
// Operand-heavy launches of 256-wide tiles run as CTA pairs (cta_group::2): two SMs
// compute one 256 x 256 tile, each loading half of its operands.
// Small-M projections whose tiles cannot fill the GPU split K, in one of two ways:
//   - cluster splits: the S parts of one output tile run as one thread-block cluster,
//     each stages its fp32 accumulator in its own shared memory, and after a cluster
//     barrier CTA rank r sums rows [r*128/S, (r+1)*128/S) of all S staged tiles in split
//     order through distributed shared memory (deterministic, no global scratch, no
//     CTA waits on a flag);
//   - deferred splits: the S parts run as independent CTAs, each storing its raw fp32
//     partial product into its own slab, and the kernel that consumes the projection
//     (the LayerNorm after a residual-stream projection) sums the slabs in split order.
// The K/V projection's kernels carry four more warps that compute the memory LayerNorm
// statistics of A's rows while the tensor cores run: jobs of 16 rows, spread over every
// CTA of the launch and paced by its producer, read from L2 just ahead of the GEMM's own
// copies of the rows (shared memory has no bandwidth to spare next to the MMAs), each
// warp publishing its 4 rows through a flag that the epilogues of every tile of those
// rows wait for before applying the fold (warps 6..9).  The rows are read from HBM once.
// Every wait (mbarrier, flag, pacing) is bounded: on a timeout the CTA sets the timeout
// flag, waits (bounded) for its own copies and MMAs in flight, frees TMEM and returns.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace clef {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kStatsWarps = 4;  // LayerNorm-statistics warps of the K/V projection's kernels
constexpr int kMaxSplits = 4;  // cluster size of a split-K tile (8-CTA clusters did not all fit at once)

struct GemmArgs {
    int n_mtiles, n_ntiles, kblocks;
    int a_rows;                    // rows of A's tensor map (a row at or past it reads as zeros)
    int splits, kb_per_split;      // split-K: each output tile's K range cut into `splits` parts,
                                   // one cluster of `splits` CTAs per output tile
    const int32_t* a_row_of_mtile;
    GemmEpilogue epi;
    int* dev_flags;
    int prefetch_b;                // B tiles of the first stages may be requested before the PDL wait
    int deferred;                  // split-K without a cluster: split sp stores its raw partial
    int64_t part_stride;           // into slab sp (elements between slabs) of the epilogue output
    const uint16_t* a_ptr;         // LN fold: A itself (row stride lda elements), read by the
    int64_t lda;                   // statistics jobs
};

// Tile t of the persistent walk: split fastest, then N, then M.
struct TileId {
    int mt, nt, sp, out;  // out = output tile index (mt * n_ntiles + nt)
};
__device__ __forceinline__ TileId decode_tile(const GemmArgs& a, int t) {
    TileId id;
    id.sp = t % a.splits;
    id.out = t / a.splits;
    id.mt = id.out / a.n_ntiles;
    id.nt = id.out % a.n_ntiles;
    return id;
}

// The it-th tile of this CTA's persistent walk.  Single CTAs: tiles t = blockIdx.x +
// it * gridDim.x.  CTA pairs: the two CTAs of a cluster take two consecutive M tiles
// of one N tile (rank r takes M tile 2 * group + r: the pair's 256-row tile) and walk
// the groups together.
template <bool PAIR>
__device__ __forceinline__ bool tile_at(const GemmArgs& a, int it, TileId& id) {
    if constexpr (!PAIR) {
        const int t = int(blockIdx.x) + it * int(gridDim.x);
        if (t >= a.n_mtiles * a.n_ntiles * a.splits) return false;
        id = decode_tile(a, t);
        return true;
    } else {
        const int g = int(blockIdx.x) / 2 + it * (int(gridDim.x) / 2);
        if (g >= (a.n_mtiles + 1) / 2 * a.n_ntiles) return false;
        id.sp = 0;
        id.nt = g % a.n_ntiles;
        id.mt = (g / a.n_ntiles) * 2 + int(blockIdx.x) % 2;
        id.out = id.mt * a.n_ntiles + id.nt;
        return true;
    }
}

// PAIR: each CTA holds its 128 A rows and half (BN / 2 rows) of the pair's B tile.
// SUB: 64-wide K slices (one 128-byte swizzle atom each) per pipeline stage.  Pairs and
// the 64- and 128-wide single-CTA tiles take two per stage, so that the single
// MMA-issuing thread waits, fences and commits once per eight MMAs instead of once per
// four (a split's last stage holds one slice when its K-slice count is odd).
// STATS: the kernel also computes the LayerNorm statistics of its A rows (the K/V
// projection with the memory LayerNorm folded in).
template <int BN, bool PAIR, bool STATS>
struct GemmCfg {
    static constexpr int THREADS = 192 + (STATS ? 32 * kStatsWarps : 0);
    static constexpr int SUB = (PAIR || BN < 256) ? 2 : 1;
    static constexpr int A_ATOM = BM * BK * 2;
    static constexpr int A_BYTES = SUB * A_ATOM;
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;
    static constexpr int B_ATOM = B_ROWS * BK * 2;
    static constexpr int B_BYTES = SUB * B_ATOM;
    static constexpr int STAGES = PAIR ? 3 : ((BN == 256) ? 4 : (BN == 128 ? 3 : 4));
    static constexpr int SMEM = STAGES * (A_BYTES + B_BYTES) + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
};

// Columns n0 .. n0 + 15 of row m; mu and rs are the row's LayerNorm statistics (LN fold).
template <int BN>
__device__ __forceinline__ void epilogue_chunk(const GemmEpilogue& e, int m, int n0, const uint32_t (&r)[16],
                                               int64_t slab, float mu, float rs) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
    if (e.kind == EPI_KV_LNFOLD) {
        // rstd == 0 marks a row of a record's round-up slack: stored as zeros, so that
        // whatever the padding held never reaches attention as a non-finite value
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = rs == 0.f ? 0.f : rs * (v[j] - mu * e.col_c[n0 + j]) + e.bias_f32[n0 + j];
    } else {
        if (e.bias_bf16) {
            const uint4* bp = reinterpret_cast<const uint4*>(e.bias_bf16 + n0);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint4 w = bp[q];
                v[q * 8 + 0] += bf16_lo(w.x); v[q * 8 + 1] += bf16_hi(w.x);
                v[q * 8 + 2] += bf16_lo(w.y); v[q * 8 + 3] += bf16_hi(w.y);
                v[q * 8 + 4] += bf16_lo(w.z); v[q * 8 + 5] += bf16_hi(w.z);
                v[q * 8 + 6] += bf16_lo(w.w); v[q * 8 + 7] += bf16_hi(w.w);
            }
        } else if (e.bias_f32) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += e.bias_f32[n0 + j];
        }
        if (e.gelu) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = gelu_exact(v[j]);
        }
    }
    if (e.kind == EPI_F32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(e.out) + slab + int64_t(m) * e.ldo + n0);
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(e.out) + int64_t(m) * e.ldo + n0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint4 w;
            w.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
            w.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
            w.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
            w.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
            o[q] = w;
        }
    }
}

// The split-K reduction's epilogue (never the LN fold): columns n0 .. n0 + 15 of row m,
// the bias read from the tile's staged copy `sbias` (column n0 at sbias[0]).
__device__ __forceinline__ void epilogue_chunk_split(const GemmEpilogue& e, int m, int n0, const float* sbias,
                                                     const float (&acc)[16]) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = acc[j] + sbias[j];
    if (e.gelu) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = gelu_exact(v[j]);
    }
    if (e.kind == EPI_F32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(e.out) + int64_t(m) * e.ldo + n0);
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(e.out) + int64_t(m) * e.ldo + n0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint4 w;
            w.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
            w.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
            w.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
            w.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
            o[q] = w;
        }
    }
}

// Memory LayerNorm statistics (mean, 1/sqrt(var + eps)) of one bf16 row of K values, by
// the 8 threads of an aligned 8-lane group (`part` = lane & 7).  The row's values are
// taken less a shift (the mean of its first 8 values, which keeps the fp32 sums free
// of cancellation for rows far from zero mean); thread `part` sums and square-sums the
// 16-byte chunks part, part + 8, ... over two interleaved accumulators, and the group
// adds its 8 partial sums in a butterfly (every lane ends with the same bits).  The
// loads go through L2 (not L1): the GEMM's own copies of the same rows follow shortly
// and find them there.
__device__ __forceinline__ float2 row_moments(const uint16_t* row, int K, int part, unsigned group_mask) {
    const uint4* rp = reinterpret_cast<const uint4*>(row);
    const uint4 h = __ldcg(rp);
    const float shift = ((bf16_lo(h.x) + bf16_hi(h.x)) + (bf16_lo(h.y) + bf16_hi(h.y)) +
                         ((bf16_lo(h.z) + bf16_hi(h.z)) + (bf16_lo(h.w) + bf16_hi(h.w)))) * 0.125f;
    float s0 = 0.f, s1 = 0.f, q0 = 0.f, q1 = 0.f;
    const int n16 = K >> 3;
#pragma unroll 8
    for (int c = part; c < n16; c += 8) {
        const uint4 v = __ldcg(rp + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float d0 = bf16_lo(w[i]) - shift, d1 = bf16_hi(w[i]) - shift;
            s0 += d0; q0 = fmaf(d0, d0, q0);
            s1 += d1; q1 = fmaf(d1, d1, q1);
        }
    }
    float s = s0 + s1, q = q0 + q1;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        s += __shfl_xor_sync(group_mask, s, o);
        q += __shfl_xor_sync(group_mask, q, o);
    }
    s /= float(K);
    q /= float(K);
    return make_float2(shift + s, rsqrtf(fmaxf(q - s * s, 0.f) + 1e-5f));
}

// PAIR (CTA pairs on cta_group::2) is only launched without split-K.
//
// CTA pairs.  Each CTA's producer loads its own A tile (128 rows) and its half of the
// pair's B tile into its own shared memory.  Rank 0 issues the pair's MMAs (M = 256),
// so every copy of both CTAs completes its bytes on rank 0's `full` barrier (rank 1
// names it through the cta_group::2 form of the copy), which rank 0's producer arms
// for both CTAs' bytes.  Rank 0's MMA thread commits every stage to the `empty`
// barriers of both CTAs and every finished accumulator to the `tfull` barriers of
// both; the epilogue warps of both CTAs arrive on rank 0's `tempty`.  Rank 1 cannot
// observe its own copies land (they complete on rank 0), so it leaves only through
// the final cluster barrier, after rank 0 has consumed or waited for every stage.
template <int BN, bool PAIR, bool STATS>
__global__ void __launch_bounds__(GemmCfg<BN, PAIR, STATS>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args) {
    using C = GemmCfg<BN, PAIR, STATS>;
    constexpr int kRedLd = BN + 4;  // staged split-K row stride (floats): conflict-free float4 rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* load_mt = abort_flag + 1;  // STATS: M tile the producer is loading (INT_MAX: done)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // rank 1 of a pair issues no MMA
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PAIR ? 2 * 4 : 4 * 32);  // pairs: one arrival per epilogue warp of each CTA
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *load_mt = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        if constexpr (PAIR) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        else tmem_alloc(tmem_slot, C::TMEM_COLS);
        tc_fence_before();
    }
    __syncthreads();
    // pairs: the peer arrives on this CTA's barriers, so both CTAs' barriers are
    // initialised (and TMEM allocated) before either goes on
    if constexpr (PAIR) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kblocks = args.kblocks;
    // When B holds weights, the producer requests the B tiles of the first stages of its
    // first tile before the dependent-launch wait: only A (and the epilogue's inputs) may
    // come from the previous kernel.  Each such stage is armed for its full A + B byte
    // count now; its A tile follows once the wait returns.
    int n_pre = 0;
    if constexpr (!PAIR) {
        TileId id0;
        if (args.prefetch_b && warp == 0 && lane == 0 && tile_at<PAIR>(args, 0, id0)) {
            const int kb0 = id0.sp * args.kb_per_split, kb1 = min(kb0 + args.kb_per_split, kblocks);
            n_pre = min(C::STAGES, (kb1 - kb0 + C::SUB - 1) / C::SUB);
            for (int i = 0; i < n_pre; ++i) {
                const int kbs = kb0 + i * C::SUB, nu = min(C::SUB, kb1 - kbs);
                mbar_arrive_expect_tx(&full[i], nu * (C::A_ATOM + C::B_ATOM));
                for (int u = 0; u < nu; ++u)
                    tma_load_2d(sB + i * C::B_BYTES + u * C::B_ATOM, &tmB, (kbs + u) * BK, id0.nt * BN, &full[i]);
            }
        }
    }
    griddep_launch();
    griddep_wait();  // operands and outputs may belong to the previous kernel of the stream

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t leader_full = PAIR ? cluster_map(smem_u32(full), 0) : 0u;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[C::STAGES];
            for (int s = 0; s < C::STAGES; ++s) armed[s] = 0;
            bool ok = true;
            TileId id;
            for (int it = 0; ok && tile_at<PAIR>(args, it, id); ++it) {
                if (STATS) *load_mt = id.mt;
                const int a_row = id.mt >= args.n_mtiles ? args.a_rows
                                  : args.a_row_of_mtile ? args.a_row_of_mtile[id.mt] : id.mt * BM;
                const int b_row = id.nt * BN + int(rank) * C::B_ROWS;  // pairs: this CTA's half of B
                const int kb0 = id.sp * args.kb_per_split, kb1 = min(kb0 + args.kb_per_split, kblocks);
                for (int kb = kb0; kb < kb1; kb += C::SUB) {
                    const int nu = PAIR ? C::SUB : min(C::SUB, kb1 - kb);  // K slices in this stage (pairs never split)
                    const bool pre = n_pre > 0;  // stage armed and its B requested before the wait
                    if (pre) {
                        --n_pre;
                    } else {
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.dev_flags)) {
                            ok = false;
                            break;
                        }
                        // pairs: rank 0's barrier counts the stage's bytes of both CTAs
                        if (rank == 0)
                            mbar_arrive_expect_tx(&full[stage], (PAIR ? 2 : 1) * nu * (C::A_ATOM + C::B_ATOM));
                    }
#pragma unroll
                    for (int u = 0; u < C::SUB; ++u) {
                        if (u >= nu) break;
                        if (PAIR && rank != 0) {
                            const uint32_t bar = leader_full + 8u * uint32_t(stage);
                            tma_load_2d_pair(sA + stage * C::A_BYTES + u * C::A_ATOM, &tmA, (kb + u) * BK, a_row, bar);
                            tma_load_2d_pair(sB + stage * C::B_BYTES + u * C::B_ATOM, &tmB, (kb + u) * BK, b_row, bar);
                        } else {
                            tma_load_2d(sA + stage * C::A_BYTES + u * C::A_ATOM, &tmA, (kb + u) * BK, a_row, &full[stage]);
                            if (!pre)
                                tma_load_2d(sB + stage * C::B_BYTES + u * C::B_ATOM, &tmB, (kb + u) * BK, b_row,
                                            &full[stage]);
                        }
                    }
                    ++armed[stage];
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (STATS) *load_mt = 0x7fffffff;
            if (!ok && rank == 0) {  // let every copy this CTA's barriers count land before it exits
                for (int s = 0; s < C::STAGES; ++s)
                    if (armed[s] != 0) mbar_wait_bounded(&full[s], (armed[s] - 1) & 1u, nullptr, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1 && PAIR && rank != 0) {
        // rank 1 of a pair issues no MMA
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
            // pairs: the peer's empty / tfull barriers (same offsets in rank 1's shared memory)
            const uint32_t peer_empty = PAIR ? cluster_map(smem_u32(empty), 1) : 0u;
            const uint32_t peer_tfull = PAIR ? cluster_map(smem_u32(tfull), 1) : 0u;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            TileId id;
            for (int it = 0; ok && tile_at<PAIR>(args, it, id); ++it, ++local) {
                const int acc = local & 1;
                const uint32_t use = uint32_t(local >> 1);
                if (!mbar_wait_bounded(&tempty[acc], (use & 1u) ^ 1u, abort_flag, args.dev_flags, kWaitLimitNs, PAIR))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
                const int kb0 = id.sp * args.kb_per_split, kb1 = min(kb0 + args.kb_per_split, kblocks);
                for (int kb = kb0; kb < kb1; kb += C::SUB) {
                    const int nu = PAIR ? C::SUB : min(C::SUB, kb1 - kb);
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.dev_flags)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors of the stage's first K slice; each 16-wide slice is 32 bytes on
                    // (2 in the descriptor's 16-byte address field)
#pragma unroll
                    for (int u = 0; u < C::SUB; ++u) {
                        if (u >= nu) break;
                        const uint64_t da = smem_desc_sw128(smem_u32(sA + stage * C::A_BYTES + u * C::A_ATOM));
                        const uint64_t db = smem_desc_sw128(smem_u32(sB + stage * C::B_BYTES + u * C::B_ATOM));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint32_t accum = (kb > kb0 || u > 0 || k > 0) ? 1u : 0u;
                            if constexpr (PAIR)
                                tc_mma_bf16_pair(d_tmem, da + uint64_t(2 * k), db + uint64_t(2 * k), idesc, accum);
                            else
                                tc_mma_bf16(d_tmem, da + uint64_t(2 * k), db + uint64_t(2 * k), idesc, accum);
                        }
                    }
                    if constexpr (PAIR) {  // the stage is free in both CTAs once the MMAs are done
                        tc_commit_pair(smem_u32(&empty[stage]));
                        tc_commit_pair(peer_empty + 8u * uint32_t(stage));
                    } else {
                        tc_commit(&empty[stage]);
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    if constexpr (PAIR) {
                        tc_commit_pair(smem_u32(&tfull[acc]));
                        tc_commit_pair(peer_tfull + 8u * uint32_t(acc));
                    } else {
                        tc_commit(&tfull[acc]);
                    }
                }
            }
            // every MMA this thread issued completes before TMEM is released
            if constexpr (PAIR) tc_commit_pair(smem_u32(drain));
            else tc_commit(drain);
            mbar_wait_bounded(drain, 0, nullptr, args.dev_flags);
        }
        __syncwarp();
    } else if (STATS && warp >= 6) {
        // LayerNorm statistics jobs: job j covers rows (j % 8) * 16 .. + 15 of 128-row tile
        // j / 8; the jobs are dealt round-robin over the launch's CTAs in tile order.  8
        // threads per row; warp w of the four publishes rows 4w .. 4w + 3 of the job.
        // Pacing: a job for tile mt starts once this CTA's producer is loading an M tile
        // of at least mt.  With the jobs dealt in tile order, each CTA's jobs then run
        // about when the GEMM reaches their rows: the rows stream in alongside the GEMM's
        // own operand copies (which find them in L2) instead of in one burst ahead of
        // them, and a job still ends well inside the mainloop of its tiles.  The rule
        // cannot deadlock: the producer's way to its first tile of M index mt or more only
        // waits on epilogues of tiles below mt, whose jobs come earlier.
        const int t = int(threadIdx.x) - 192;
        const int part = t & 7;
        const unsigned group_mask = 0xffu << (lane & 24);
        const int n_jobs = args.n_mtiles * 8;
        bool ok = true;
        for (int j = int(blockIdx.x); ok && j < n_jobs; j += int(gridDim.x)) {
            const int mt = j >> 3, r = (j & 7) * 16 + (t >> 3), m = mt * BM + r;
            const uint64_t t0 = global_ns();
            while (*load_mt < mt) {  // each lane on its own, then all lanes agree
                if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
                    ok = false;
                    break;
                }
                __nanosleep(256);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            bool real = m < args.epi.M;
            if (real && args.epi.tile_rec) {
                const int b = args.epi.tile_rec[mt];
                real = m - args.epi.rec_row_off[b] < args.epi.rec_len[b];
            }
            float2 st = make_float2(0.f, 0.f);  // padding rows: mu = rstd = 0
            if (real) {
                const int64_t a_row = (args.a_row_of_mtile ? args.a_row_of_mtile[mt] : mt * BM) + r;
                st = row_moments(args.a_ptr + a_row * args.lda, args.kblocks * BK, part, group_mask);
            }
            if (part == 0 && m < args.epi.M) {
                args.epi.row_mu[m] = st.x;
                args.epi.row_rstd[m] = st.y;
                __threadfence();  // the rows' statistics reach GPU scope before the flag
            }
            __syncwarp();
            if (lane == 0) flag_publish(args.epi.row_flags + (j * 4 + (warp - 6)), args.epi.epoch);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(args.dev_flags, kFlagTimeout);
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may read
        const int r_in_tile = quarter * 32 + lane;
        // pairs: rank 0's tempty barriers, where the epilogue warps of both CTAs arrive
        const uint32_t leader_tempty = PAIR ? cluster_map(smem_u32(tempty), 0) : 0u;
        int local = 0;
        TileId id;
        for (int it = 0; tile_at<PAIR>(args, it, id); ++it, ++local) {
            const int acc = local & 1;
            const uint32_t use = uint32_t(local >> 1);
            // split-K: this thread's share of the tile's bias, read while the MMAs run
            float bias_share[(BN + 127) / 128];
            if (args.splits > 1 && !args.deferred) {
#pragma unroll
                for (int k = 0; k < (BN + 127) / 128; ++k) {
                    const int j = (threadIdx.x - 64) + 128 * k, n = id.nt * BN + j;
                    bias_share[k] = j >= BN ? 0.f
                                    : args.epi.bias_bf16 ? bf16_to_float(args.epi.bias_bf16[n])
                                    : (args.epi.bias_f32 ? args.epi.bias_f32[n] : 0.f);
                }
            }
            int ok = 1;
            if (lane == 0) ok = mbar_wait_bounded(&tfull[acc], use & 1u, abort_flag, args.dev_flags) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int m = id.mt * BM + r_in_tile;
            const bool store = m < args.epi.M;
            float row_mu = 0.f, row_rs = 0.f;
            if constexpr (STATS) {  // this row's LayerNorm statistics, once its job has published them
                const bool got = !store || flag_wait_bounded(args.epi.row_flags + (m >> 2), args.epi.epoch,
                                                             abort_flag, args.dev_flags);
                if (!__all_sync(0xffffffffu, got)) break;
                if (store) {
                    row_mu = __ldcg(args.epi.row_mu + m);
                    row_rs = __ldcg(args.epi.row_rstd + m);
                }
            }
            if (args.splits == 1 || args.deferred) {
                const int64_t slab = args.deferred ? int64_t(id.sp) * args.part_stride : 0;
#pragma unroll 1
                for (int c = 0; c < BN / 16; ++c) {
                    uint32_t r[16];
                    tmem_ld16(tmem_base + uint32_t(acc * BN + c * 16) + (uint32_t(quarter * 32) << 16), r);
                    tmem_ld_wait();
                    if (store) epilogue_chunk<BN>(args.epi, m, id.nt * BN + c * 16, r, slab, row_mu, row_rs);
                }
                tc_fence_before();
                if constexpr (PAIR) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(leader_tempty + 8u * uint32_t(acc));
                } else {
                    mbar_arrive(&tempty[acc]);
                }
                continue;
            }
            // split-K: stage this split's fp32 rows in shared memory.  The operand stages
            // are idle by now: a split CTA has one tile, whose MMAs have all completed.
            float* red = reinterpret_cast<float*>(smem) + r_in_tile * kRedLd;
#pragma unroll 1
            for (int c = 0; c < BN / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(tmem_base + uint32_t(acc * BN + c * 16) + (uint32_t(quarter * 32) << 16), r);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<float4*>(red + c * 16 + 4 * q) =
                        make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                    __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            float* sbias = reinterpret_cast<float*>(smem) + BM * kRedLd;  // after the staged rows
#pragma unroll
            for (int k = 0; k < (BN + 127) / 128; ++k) {
                const int j = (threadIdx.x - 64) + 128 * k;
                if (j < BN) sbias[j] = bias_share[k];
            }
        }
    }
    if (!PAIR && !STATS && args.splits > 1 && !args.deferred) {
        // every thread of every CTA of the cluster passes both barriers, on every path
        cluster_sync();
        if (warp >= 2) {
            const TileId id = decode_tile(args, blockIdx.x);
            const int S = args.splits, rows = BM / S;
            constexpr int chunks = BN / 16;
            const uint32_t red0 = smem_u32(smem);
            const float* sbias = reinterpret_cast<const float*>(smem) + BM * kRedLd;
#pragma unroll 1
            for (int i = threadIdx.x - 64; i < rows * chunks; i += 128) {
                const int row = id.sp * rows + i / chunks, c = i % chunks;
                const uint32_t off = red0 + uint32_t((row * kRedLd + c * 16) * 4);
                const int m = id.mt * BM + row;
                const int n0 = id.nt * BN + c * 16;
                // every split's slice is requested before any is added (one round trip),
                // then the slices are summed in split order
                float4 w[kMaxSplits][4];
#pragma unroll
                for (int sp = 0; sp < kMaxSplits; ++sp) {
                    if (sp < S) {
                        const uint32_t a = cluster_map(off, uint32_t(sp));
#pragma unroll
                        for (int q = 0; q < 4; ++q) w[sp][q] = ld_cluster_f4(a + 16u * q);
                    }
                }
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
                for (int sp = 0; sp < kMaxSplits; ++sp) {
                    if (sp < S) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            v[4 * q] += w[sp][q].x; v[4 * q + 1] += w[sp][q].y;
                            v[4 * q + 2] += w[sp][q].z; v[4 * q + 3] += w[sp][q].w;
                        }
                    }
                }
                if (m < args.epi.M) epilogue_chunk_split(args.epi, m, n0, sbias + c * 16, v);
            }
        }
        cluster_sync();  // no CTA leaves while another may still read its shared memory
    }
    __syncthreads();
    // pairs: no CTA leaves (or frees TMEM) while rank 0's MMAs may still read its shared
    // memory or write its TMEM, or while its peer may still arrive on its barriers
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

bool make_tma_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_elems,
                      uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_elems * 2};
    cuuint32_t box[2] = {uint32_t(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Opts the kernel into its dynamic shared memory size (once per instantiation).
template <int BN, bool PAIR, bool STATS>
cudaError_t kernel_attributes() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_tc_kernel<BN, PAIR, STATS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   GemmCfg<BN, PAIR, STATS>::SMEM);
    });
    return err;
}

// How many clusters of `size` CTAs of this kernel the GPU holds at once (0: none).
template <int BN, bool PAIR, bool STATS>
int active_clusters(int size) {
    if (kernel_attributes<BN, PAIR, STATS>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(size);
    cfg.blockDim = dim3(GemmCfg<BN, PAIR, STATS>::THREADS);
    cfg.dynamicSmemBytes = GemmCfg<BN, PAIR, STATS>::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, PAIR, STATS>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Largest cluster size S (power of two, at most kMaxSplits) of which the GPU can hold
// at least one cluster of this kernel.
template <int BN>
int max_cluster_splits() {
    static std::once_flag once;
    static int best = 1;
    std::call_once(once, [] {
        for (int S = kMaxSplits; S > 1; S >>= 1) {
            if (active_clusters<BN, false, false>(S) > 0) {
                best = S;
                break;
            }
        }
    });
    return best;
}

// CTA pairs of the BN = 256 pair kernel the GPU holds at once (0: the mode is unavailable).
template <bool STATS>
int pair_clusters() {
    static std::once_flag once;
    static int n = 0;
    std::call_once(once, [] { n = active_clusters<256, true, STATS>(2); });
    return n;
}

cudaError_t launch_cluster(void (*kernel)(CUtensorMap, CUtensorMap, GemmArgs), int grid, int cluster, int threads,
                           size_t smem, cudaStream_t s, const CUtensorMap& ta, const CUtensorMap& tb,
                           const GemmArgs& a) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return counted(cudaLaunchKernelEx(&cfg, kernel, ta, tb, a));
}

// Operand-heavy BN = 256 launches (more output tiles than SMs) run as CTA pairs: the
// pair's 256 x 256 tile is one cta_group::2 MMA stream, and each CTA loads only its own
// 128 A rows and 128 of the 256 B rows, which cuts the L2-to-SM operand traffic per K
// block from 48 KB to 32 KB per CTA.  Returns false (nothing launched) when the GPU
// cannot hold a pair of this kernel.
template <bool STATS>
bool launch_pair(const GemmProblem& p, const GemmArgs& a, cudaStream_t s, const CUtensorMap& ta, cudaError_t* err) {
    using C = GemmCfg<256, true, STATS>;
    const int clusters = pair_clusters<STATS>();
    if (clusters <= 0) return false;
    CUtensorMap tbh;  // B in 128-row boxes: this CTA's half of the pair's B tile
    if (!make_tma_2d_bf16(&tbh, p.B, uint64_t(p.K), uint64_t(p.N), uint64_t(p.ldb), C::B_ROWS)) {
        *err = cudaErrorInvalidValue;
        return true;
    }
    const int groups = (a.n_mtiles + 1) / 2 * a.n_ntiles;
    const int grid = 2 * std::min(groups, clusters);
    *err = launch_cluster(gemm_tc_kernel<256, true, STATS>, grid, 2, C::THREADS, C::SMEM, s, ta, tbh, a);
    return true;
}

template <int BN, bool STATS>
cudaError_t launch_bn(const GemmProblem& p, const GemmEpilogue& e, int* flags, cudaStream_t s, int splits,
                      bool deferred = false) {
    using C = GemmCfg<BN, false, STATS>;
    const cudaError_t attr_err = kernel_attributes<BN, false, STATS>();
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap ta, tb;
    if (!make_tma_2d_bf16(&ta, p.A, uint64_t(p.K), uint64_t(p.a_rows), uint64_t(p.lda), BM)) return cudaErrorInvalidValue;
    GemmArgs a;
    a.n_mtiles = p.n_mtiles;
    a.n_ntiles = p.N / BN;
    a.kblocks = p.K / BK;
    a.a_rows = int(p.a_rows);
    a.splits = splits;
    a.kb_per_split = a.kblocks / splits;
    a.a_row_of_mtile = p.a_row_of_mtile;
    a.epi = e;
    a.dev_flags = flags;
    a.prefetch_b = p.b_is_weight ? 1 : 0;
    a.deferred = deferred ? 1 : 0;
    a.part_stride = p.part_stride;
    a.a_ptr = p.A;
    a.lda = p.lda;
    const int sms = num_sms();
    const int out_tiles = a.n_mtiles * a.n_ntiles;
    const int tiles = out_tiles * a.splits;
    if constexpr (BN == 256) {
        if (a.splits == 1 && !deferred && out_tiles > sms) {
            a.prefetch_b = 0;
            cudaError_t err = cudaSuccess;
            if (launch_pair<STATS>(p, a, s, ta, &err)) return err;
            a.prefetch_b = p.b_is_weight ? 1 : 0;
        }
    }
    if (!make_tma_2d_bf16(&tb, p.B, uint64_t(p.K), uint64_t(p.N), uint64_t(p.ldb), BN)) return cudaErrorInvalidValue;
    if (a.splits > 1 && !deferred)  // one CTA per (output tile, split); the splits of a tile form one cluster
        return launch_cluster(gemm_tc_kernel<BN, false, STATS>, tiles, a.splits, C::THREADS, C::SMEM, s, ta, tb, a);
    const int grid = tiles < sms ? tiles : sms;
    return launch_pdl(gemm_tc_kernel<BN, false, STATS>, dim3(grid), dim3(C::THREADS), C::SMEM, s, ta, tb, a);
}

}  // namespace

std::atomic<uint64_t> g_kernel_launches{0};

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

// Deferred split-K: no cluster reduction, so a split costs only its slab (written by the
// GEMM, read back by the consumer through L2, about 8 TB/s each way), and any divisor of
// the K blocks that leaves at least 4 blocks per split may serve.  Otherwise the same
// estimate as the cluster splits below: operand tiles from L2 at about 11 TB/s into CTAs
// that each take in about 90 GB/s.
void partial_split_config(int n_mtiles, int N, int K, int* bn_out, int* splits_out) {
    const int sms = num_sms();
    const int kblocks = K / BK;
    double best = 1e30;
    int bn = 64, splits = 1;
    for (int w : {64, 128, 256}) {
        if (N % w) continue;
        const int tiles = n_mtiles * (N / w);
        for (int S = 1; S <= kblocks; ++S) {
            if (kblocks % S || (S > 1 && kblocks / S < 4) || tiles * S > 2 * sms) continue;
            const int ctas = std::min(tiles * S, sms);
            const int waves = (tiles * S + sms - 1) / sms;
            const double per_cta = double(waves) * (kblocks / S) * (BM + w) * BK * 2.0;
            const double slabs = 2.0 * S * n_mtiles * double(BM) * N * 4.0;
            const double t = std::max(per_cta / 90e3, per_cta * ctas / 11e6) + slabs / 8e6;
            if (t < best) {
                best = t;
                bn = w;
                splits = S;
            }
        }
    }
    *bn_out = bn;
    *splits_out = splits;
}

cudaError_t launch_gemm(const GemmProblem& p, const GemmEpilogue& e, int* dev_flags, cudaStream_t s, int force_bn) {
    if (p.n_mtiles <= 0 || p.N <= 0) return cudaSuccess;
    if (p.K % BK != 0 || p.N % 64 != 0 || p.lda % 8 != 0 || p.ldb % 8 != 0) return cudaErrorInvalidValue;
    if (p.defer_splits > 0) {
        if (e.kind != EPI_F32 || e.gelu || e.bias_bf16 || e.bias_f32 || (p.K / BK) % p.defer_splits ||
            p.N % p.defer_bn)
            return cudaErrorInvalidValue;
        switch (p.defer_bn) {
            case 256: return launch_bn<256, false>(p, e, dev_flags, s, p.defer_splits, true);
            case 128: return launch_bn<128, false>(p, e, dev_flags, s, p.defer_splits, true);
            case 64: return launch_bn<64, false>(p, e, dev_flags, s, p.defer_splits, true);
            default: return cudaErrorInvalidValue;
        }
    }
    if (e.kind == EPI_KV_LNFOLD) {
        // the LN fold computes its row statistics in the kernel: never split, every row's
        // output tiles see its whole K range
        if (p.allow_split || !e.row_mu || !e.row_rstd || !e.row_flags) return cudaErrorInvalidValue;
        const int sms = num_sms();
        int bn = force_bn;
        if (bn == 0) {
            bn = 64;
            if (p.N % 256 == 0 && p.n_mtiles * (p.N / 256) >= sms) bn = 256;
            else if (p.N % 128 == 0 && p.n_mtiles * (p.N / 128) >= sms) bn = 128;
        }
        if (p.N % bn != 0) return cudaErrorInvalidValue;
        static std::atomic<uint64_t> epochs{0};
        GemmEpilogue ef = e;
        ef.epoch = epochs.fetch_add(1, std::memory_order_relaxed) + 1;  // never 0, the cleared value
        switch (bn) {
            case 256: return launch_bn<256, true>(p, ef, dev_flags, s, 1);
            case 128: return launch_bn<128, true>(p, ef, dev_flags, s, 1);
            default: return launch_bn<64, true>(p, ef, dev_flags, s, 1);
        }
    }
    const int sms = num_sms();
    const int kblocks = p.K / BK;
    int bn = force_bn, splits = 1;
    if (bn == 0 && !p.allow_split) {
        bn = 64;
        if (p.N % 256 == 0 && p.n_mtiles * (p.N / 256) >= sms) bn = 256;
        else if (p.N % 128 == 0 && p.n_mtiles * (p.N / 128) >= sms) bn = 128;
    } else if (bn == 0) {
        // Small-M projections: pick the tile width and the split count with the least
        // estimated time.  A launch streams its operand tiles from L2 (aggregate about
        // 11 TB/s) into CTAs that each take in about 90 GB/s with this pipeline depth;
        // a split costs about 2 us of cluster barriers and reduction.  The constants
        // come from sweeping every (width, split) of the head's projections on GB300.
        double best = 1e30;
        for (int w : {64, 128, 256}) {
            if (p.N % w) continue;
            const int tiles = p.n_mtiles * (p.N / w);
            const int max_s = w == 64 ? max_cluster_splits<64>() : (w == 128 ? max_cluster_splits<128>()
                                                                               : max_cluster_splits<256>());
            for (int S = 1; S <= 4 && S <= max_s; S *= 2) {
                if (S > 1 && (kblocks % S || kblocks / S < 8 || tiles * S > sms)) continue;
                const int ctas = std::min(tiles * S, sms);
                const int waves = (tiles * S + sms - 1) / sms;
                const double per_cta = double(waves) * (kblocks / S) * (BM + w) * BK * 2.0;
                const double t = std::max(per_cta / 90e3, per_cta * ctas / 11e6) + (S > 1 ? 2.0 : 0.0);
                if (t < best) {
                    best = t;
                    bn = w;
                    splits = S;
                }
            }
        }
    }
    if (p.N % bn != 0) return cudaErrorInvalidValue;
    switch (bn) {
        case 256: return launch_bn<256, false>(p, e, dev_flags, s, splits);
        case 128: return launch_bn<128, false>(p, e, dev_flags, s, splits);
        default: return launch_bn<64, false>(p, e, dev_flags, s, splits);
    }
}

}  // namespace clef
