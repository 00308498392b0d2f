// Routing cross-attention of the EvidenceRoutingLayers ("clef-4bit JointSchemaHead
// walkthrough" section 3 step 2: every option is a query over the whole memory),
// split over the memory length (flash-decoding style) and merged afterwards.
//
// Work = (head, unit), unit = (record chunk of kAttnChunk memory rows, block of 64
// option queries of that record); only the blocks a record needs are listed.  The
// kernel is persistent: each CTA walks work w = blockIdx.x + i * gridDim.x (head
// fastest, so CTAs running side by side read the same memory rows).  A producer warp
// streams 64-row K and V tiles with TMA (128-byte swizzle) through a 4-stage mbarrier
// ring that runs on from one work item to the next, and loads each item's queries
// into the query slot as soon as the consumers have copied the previous item's
// queries into registers.  Four consumer warps each own 16 queries and run QK^T and
// PV on mma.sync bf16 tensor cores with an fp32 online softmax in the exp2 domain.
// Keys at or past the chunk end are masked.  Every (option, head, chunk) leaves
// (running max, running sum, unnormalised accumulator); the merge kernel rescales and
// sums the chunks.
// Every mbarrier wait is bounded; on a timeout the CTA flags it and returns.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "head_kernels.h"
#include "kernels.h"

namespace clef {

namespace {

constexpr int kKT = 64;                     // keys per tile
constexpr int kStages = 4;
constexpr int kQSlots = 1;                  // query slots: the consumers hold an item's queries in registers
constexpr int kQRows = kAttnQRows;          // option queries per work item (4 consumer warps x 16)
constexpr int kTileBytes = kKT * 128;       // [64 rows][64 bf16]
constexpr int kQBytes = kQRows * 128;
constexpr int kSmem = kQSlots * kQBytes + kStages * 2 * kTileBytes + 1024 + 128;
constexpr int kThreads = 160;               // 4 consumer warps + 1 producer warp
constexpr int kBlocksPerSM = 3;

// byte offset of 16-byte chunk `chunk` of row `row` in a tile written by TMA with the
// 128-byte swizzle (chunk index XOR row mod 8, tile base 1024-byte aligned)
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

struct Work {
    int h, qp, b, kc, o_base, O_b, t0, t1, n_tiles, kv_row0;
};

__device__ __forceinline__ Work work_of(const RouteAttnArgs& a, int w) {
    Work k;
    k.h = w % a.heads;
    const int u = w / a.heads;
    const int cx = a.unit_cx[u];
    k.qp = a.unit_qp[u];
    k.b = a.chunk_rec[cx];
    k.kc = a.chunk_idx[cx];
    k.o_base = a.rec_o_off[k.b];
    k.O_b = a.rec_o_off[k.b + 1] - k.o_base;
    const int L = a.lengths[k.b];
    k.t0 = k.kc * kAttnChunk;
    k.t1 = min(k.t0 + kAttnChunk, L);
    k.n_tiles = (k.t1 - k.t0 + kKT - 1) / kKT;
    k.kv_row0 = a.rec_row_off[k.b] + k.t0;
    return k;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, kBlocksPerSM)
    route_attn_partial_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                              const RouteAttnArgs a) {
    griddep_wait();
    griddep_launch();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                        // query slots
    uint8_t* sKV = smem + kQSlots * kQBytes;   // stage s: K at s * 2 * kTileBytes, V right after
    uint64_t* full = reinterpret_cast<uint64_t*>(sKV + kStages * 2 * kTileBytes);
    uint64_t* empty = full + kStages;
    uint64_t* qfull = empty + kStages;
    uint64_t* qempty = qfull + kQSlots;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(qempty + kQSlots);

    const int n_work = a.n_units * a.heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        for (int q = 0; q < kQSlots; ++q) {
            mbar_init(&qfull[q], 1);
            mbar_init(&qempty[q], 4);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 4) {  // producer
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmKV);
            uint32_t armed[kStages] = {};
            uint32_t armed_q[kQSlots] = {};
            int stage = 0, qs = 0;
            uint32_t phase = 0, qphase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
                const Work k = work_of(a, w);
                if (!mbar_wait_bounded(&qempty[qs], qphase ^ 1u, abort_flag, a.flags)) break;
                mbar_arrive_expect_tx(&qfull[qs], kQBytes);
                tma_load_2d(sQ + qs * kQBytes, &tmQ, k.h * 64, k.o_base + k.qp * kQRows, &qfull[qs]);
                ++armed_q[qs];
                if (++qs == kQSlots) {
                    qs = 0;
                    qphase ^= 1u;
                }
                for (int kt = 0; kt < k.n_tiles; ++kt) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.flags)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], 2 * kTileBytes);
                    uint8_t* dst = sKV + stage * 2 * kTileBytes;
                    const int row = k.kv_row0 + kt * kKT;
                    tma_load_2d(dst, &tmKV, a.k_col + k.h * 64, row, &full[stage]);
                    tma_load_2d(dst + kTileBytes, &tmKV, a.v_col + k.h * 64, row, &full[stage]);
                    ++armed[stage];
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy this thread started lands before the CTA can exit
            for (int q = 0; q < kQSlots; ++q)
                if (armed_q[q]) mbar_wait_bounded(&qfull[q], (armed_q[q] - 1) & 1u, nullptr, nullptr);
            for (int s = 0; s < kStages; ++s)
                if (armed[s]) mbar_wait_bounded(&full[s], (armed[s] - 1) & 1u, nullptr, nullptr);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int g = lane >> 2, tq = lane & 3;
    const int wrow0 = warp * 16;
    const float sl2 = a.scale_log2;
    int stage = 0, qs = 0;
    uint32_t phase = 0, qphase = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
        const Work k = work_of(a, w);
        const bool active = k.qp * kQRows + wrow0 < k.O_b;
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(&qfull[qs], qphase, abort_flag, a.flags) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return;
        uint32_t qa[4][4];
        if (active) {
            const uint32_t qb = smem_u32(sQ + qs * kQBytes);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) ldmatrix_x4(qa[ks], qb + swz(wrow0 + (lane & 15), ks * 2 + (lane >> 4)));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[qs]);  // the queries are in registers
        if (++qs == kQSlots) {
            qs = 0;
            qphase ^= 1u;
        }
        float m_r[2] = {-INFINITY, -INFINITY};
        float acc[8][4];
        // running sums of P per row, from an extra MMA of P against an all-ones block:
        // lsum[0..1] row g, lsum[2..3] row g + 8 (the n columns are equal)
        float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

        for (int kt = 0; kt < k.n_tiles; ++kt) {
            if (lane == 0) ok = mbar_wait_bounded(&full[stage], phase, abort_flag, a.flags) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) return;
            if (active) {
                const uint32_t kb = smem_u32(sKV + stage * 2 * kTileBytes);
                const uint32_t vb = kb + kTileBytes;
                float s[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                    for (int jp = 0; jp < 4; ++jp) {  // pairs of 8-key n-tiles
                        uint32_t kr[4];
                        ldmatrix_x4(kr, kb + swz(jp * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)));
                        mma_bf16_16816(s[2 * jp], qa[ks], kr[0], kr[1]);
                        mma_bf16_16816(s[2 * jp + 1], qa[ks], kr[2], kr[3]);
                    }
                }
                const int kbase = k.t0 + kt * kKT;
                if (kbase + kKT > k.t1) {  // only the chunk's last tile can hold keys past its end
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (kbase + j * 8 + tq * 2 + (c & 1) >= k.t1) s[j][c] = -INFINITY;
                }
                // raw-score row maxima; the scale is applied once per row and fused into the
                // exponent below (p = 2^(s * scale - m))
                float mx[2];
                #pragma unroll
                for (int r = 0; r < 2; ++r) {  // 16 values of row g (r = 0) or g + 8 (r = 1): a 3-input max tree
                    const int c0 = 2 * r;
                    const float a = fmax3(s[0][c0], s[0][c0 + 1], s[1][c0]), b = fmax3(s[1][c0 + 1], s[2][c0], s[2][c0 + 1]);
                    const float c = fmax3(s[3][c0], s[3][c0 + 1], s[4][c0]), d = fmax3(s[4][c0 + 1], s[5][c0], s[5][c0 + 1]);
                    const float e = fmax3(s[6][c0], s[6][c0 + 1], s[7][c0]);
                    mx[r] = fmaxf(fmax3(a, b, c), fmax3(d, e, s[7][c0 + 1]));
                }
                // The row's reference maximum m moves only when a tile's maximum exceeds it by
                // more than 2^8 (p never exceeds 2^8, so nothing overflows); the accumulator and
                // the running sum are rescaled only then, which after the first tile is rare.
                float nm[2];
                bool need[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                    mx[r] *= sl2;
                    need[r] = mx[r] > m_r[r] + 8.f;
                }
                if (__any_sync(0xffffffffu, need[0] || need[1])) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float mn = need[r] ? mx[r] : m_r[r];
                        const float corr = ex2_approx(m_r[r] - mn);
                        m_r[r] = mn;
                        lsum[2 * r] *= corr;
                        lsum[2 * r + 1] *= corr;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            acc[j][2 * r] *= corr;
                            acc[j][2 * r + 1] *= corr;
                        }
                    }
                }
                nm[0] = -m_r[0];
                nm[1] = -m_r[1];
                uint32_t pa[4][4];
                // p = 2^(s * scale - m), the exponent rounded to bf16 and raised two at a time
                // on the bf16x2 path: P feeds the bf16 P V product either way, and a rounding
                // of the exponent by 2^-9 relative changes p by at most about 7e-4 of the row
                // maximum (it grows with |s - m| while p shrinks as 2^-|s - m|)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    pa[j >> 1][(j & 1) * 2 + 0] =
                        ex2_bf16x2(pack_bf16(fmaf(s[j][0], sl2, nm[0]), fmaf(s[j][1], sl2, nm[0])));
                    pa[j >> 1][(j & 1) * 2 + 1] =
                        ex2_bf16x2(pack_bf16(fmaf(s[j][2], sl2, nm[1]), fmaf(s[j][3], sl2, nm[1])));
                }
                constexpr uint32_t kOnes = 0x3F803F80u;  // two bf16 1.0
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                    for (int dp = 0; dp < 4; ++dp) {  // pairs of 8-dim n-tiles
                        uint32_t vr[4];
                        ldmatrix_x4_trans(vr, vb + swz(ks * 16 + (lane & 15), dp * 2 + (lane >> 4)));
                        mma_bf16_16816(acc[2 * dp], pa[ks], vr[0], vr[1]);
                        mma_bf16_16816(acc[2 * dp + 1], pa[ks], vr[2], vr[3]);
                    }
                    mma_bf16_16816(lsum, pa[ks], kOnes, kOnes);  // the rows of P summed
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!active) continue;
        const float l_r[2] = {lsum[0], lsum[2]};
        const int64_t part_base = a.rec_part_off[k.b] + (int64_t(k.kc) * a.heads + k.h) * k.O_b;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int o = k.qp * kQRows + wrow0 + g + r * 8;
            if (o < k.O_b) {
                const int64_t pi = part_base + o;
                if (tq == 0) {
                    a.pm[pi] = m_r[r];
                    a.pl[pi] = l_r[r];
                }
                float* dst = a.pacc + pi * 64;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float2*>(dst + j * 8 + tq * 2) = make_float2(acc[j][2 * r], acc[j][2 * r + 1]);
            }
        }
    }
}

// Merge of the split-L partials of one (option, head): one warp, 2 dims per lane.
__global__ void __launch_bounds__(256) route_attn_merge_kernel(const RouteAttnArgs a, int O) {
    griddep_wait();
    griddep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = blockIdx.x * 8 + warp;
    if (item >= O * a.heads) return;
    const int o = item / a.heads, h = item % a.heads;
    const int b = a.o_rec[o];
    const int o_base = a.rec_o_off[b];
    const int O_b = a.rec_o_off[b + 1] - o_base;
    const int nch = (a.lengths[b] + kAttnChunk - 1) / kAttnChunk;
    const int64_t p0 = a.rec_part_off[b] + int64_t(h) * O_b + (o - o_base);  // chunk k at p0 + k * heads * O_b
    const int64_t pstride = int64_t(a.heads) * O_b;
    // Chunks in groups of 8: every load of a group (lane k: chunk k's maximum and sum;
    // all lanes: two dims of each chunk's accumulator) is issued before any is used, so
    // a group costs one round trip; groups after the first rescale what came before.
    float M = -INFINITY, Ls = 0.f, x0 = 0.f, x1 = 0.f;
    for (int k0 = 0; k0 < nch; k0 += 8) {
        const int nk = min(8, nch - k0);
        float pmk = -INFINITY, plk = 0.f;
        if (lane < nk) {
            pmk = a.pm[p0 + (k0 + lane) * pstride];
            plk = a.pl[p0 + (k0 + lane) * pstride];
        }
        float2 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = j < nk ? *reinterpret_cast<const float2*>(a.pacc + (p0 + (k0 + j) * pstride) * 64 + lane * 2)
                          : make_float2(0.f, 0.f);
        const float nm = fmaxf(M, warp_max(pmk));
        const float corr = exp2f(M - nm);  // 0 for the first group
        const float w = lane < nk ? exp2f(pmk - nm) : 0.f;
        Ls = Ls * corr + warp_sum(plk * w);
        x0 *= corr;
        x1 *= corr;
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // chunks in order; the weights come from their lanes
            const float wj = __shfl_sync(0xffffffffu, w, j);
            x0 += v[j].x * wj;
            x1 += v[j].y * wj;
        }
        M = nm;
    }
    const float inv = 1.0f / Ls;
    *reinterpret_cast<uint32_t*>(a.out + int64_t(o) * a.ldo + h * 64 + lane * 2) = pack_bf16(x0 * inv, x1 * inv);
}

cudaError_t launch_route_attn_partial(const RouteAttnArgs& a, int O, cudaStream_t s) {
    if (a.n_units <= 0 || O <= 0) return cudaSuccess;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int resident = 0;  // CTAs per SM that fit
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(route_attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (attr_err == cudaSuccess)
            attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, route_attn_partial_kernel, kThreads, kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tq, tkv;
    if (!make_tma_2d_bf16(&tq, a.q, uint64_t(a.heads) * 64, uint64_t(O), uint64_t(a.ldq), 64))
        return cudaErrorInvalidValue;
    if (!make_tma_2d_bf16(&tkv, a.kv, uint64_t(a.ldkv), uint64_t(a.kv_rows), uint64_t(a.ldkv), 64))
        return cudaErrorInvalidValue;
    const int64_t n_work = int64_t(a.n_units) * a.heads;
    if (n_work >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    const int64_t slots = int64_t(std::max(resident, 1)) * num_sms();
    const int grid = int(std::min(n_work, slots));
    return launch_pdl(route_attn_partial_kernel, dim3(unsigned(grid)), dim3(kThreads), kSmem, s, tq, tkv, a);
}

cudaError_t launch_route_attn_merge(const RouteAttnArgs& a, int O, cudaStream_t s) {
    if (O <= 0) return cudaSuccess;
    return launch_pdl(route_attn_merge_kernel, dim3((O * a.heads + 7) / 8), dim3(256), 0, s, a, O);
}

}  // namespace clef
