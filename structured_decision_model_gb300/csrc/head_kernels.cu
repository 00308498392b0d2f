// The head's non-GEMM kernels: span pooling, LayerNorm of
// the option / field streams, split-L routing attention and its merge, field
// aggregation, field self-attention, scorer input assembly, scoring with the
// per-question softmax, and the weight-preparation kernels.
#include <algorithm>

#include "common.cuh"
#include "head_kernels.h"
#include "kernels.h"

namespace clef {

// fp16 rows [rows][H] (row stride ld_src) rounded to a dense bf16 copy [rows][H]: the
// streaming path's fp16 input, 8 values (16 bytes) per thread.
__global__ void __launch_bounds__(256) f16_rows_to_bf16_kernel(const uint16_t* __restrict__ src, int64_t ld_src,
                                                              int rows, int H, uint16_t* __restrict__ dst) {
    griddep_wait();
    griddep_launch();
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int c8 = H >> 3;
    if (i >= int64_t(rows) * c8) return;
    const int64_t r = i / c8;
    const int c = int(i % c8);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * ld_src) + c);
    reinterpret_cast<uint4*>(dst + r * H)[c] = f16x8_to_bf16x8(v);
}

// Zeroes K/V rows L_b .. roundup(L_b, 128) - 1 of every record (one CTA per record).
__global__ void __launch_bounds__(256) zero_slack_kernel(uint16_t* __restrict__ kv, int ldkv,
                                                        const int32_t* __restrict__ rec_row_off,
                                                        const int32_t* __restrict__ lengths) {
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.x;
    const int L = lengths[b];
    const int slack = (L + 127) / 128 * 128 - L;
    uint4* base = reinterpret_cast<uint4*>(kv + (int64_t(rec_row_off[b]) + L) * ldkv);
    const int n = slack * (ldkv / 8);
    for (int i = threadIdx.x; i < n; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
}

// =====================================================================
// Span pooling ("clef-4bit JointSchemaHead walkthrough" section 3 step 1,
// "clef-flash-CoreAI metadata.json" decision.spans / head.reads / head.lexical).
// One CTA per work item:
//   kind 0, question q:  u_q = mean over the instruction span of LN(h_t)
//   kind 1, option j:    c_j = mean over its span of LN(h_t);  x_j = mean of lexical rows of its ids
//   kind 2, record b:    g_b = LN(h_{L_b - 1})
// LN(h_t) = (h_t - mu_t) * rstd_t * gamma + beta; the mean of the normalised rows is
// taken first and the affine part applied once.  Each thread owns 8 columns per
// step (one 16-byte load per row).  RAW = true writes plain span sums of the raw
// rows instead (the bit-exact index check).  F16 = true reads fp16 hidden rows and
// rounds each value to bf16 first, so that pooling sees the same rows as the K/V
// projection of the fp16 streaming path.
// =====================================================================
template <bool RAW, bool F16>
__global__ void __launch_bounds__(256, 3) span_pool_kernel(SpanPoolArgs a) {
    griddep_wait();
    griddep_launch();
    // the item, its record and its span in one 16-byte load (no dependent table lookups)
    const int4 it = a.items[blockIdx.x];
    const int kind = int(uint32_t(it.x) >> 30);
    const int idx = it.x & ((1 << 30) - 1);
    const int H = a.H;
    const int n8 = H >> 3;
    const int b = it.y, s = it.z, e = it.w;
    const int64_t rec_base = int64_t(b) * a.Lpad;
    const int stat_base = a.rec_row_off[b];
    const float inv_n = 1.0f / float(e - s);
    for (int c8 = threadIdx.x; c8 < n8; c8 += blockDim.x) {
        float acc[8], lex[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) { acc[k] = 0.f; lex[k] = 0.f; }
        // rows in groups of 6: all loads of a group are issued before its sums, which are
        // then taken in row order (the same order as one row at a time); the hidden rows and
        // the lexical rows of an option span are two separate passes (fewer live registers).
        // Groups of 6 at 3 CTAs per SM measured fastest (groups of 4, 6, 8 at 2-4 CTAs).
        for (int t0 = s; t0 < e; t0 += 6) {
            const int nr = min(6, e - t0);
            uint4 w[6];
            float m[6], rs[6];
#pragma unroll
            for (int u = 0; u < 6; ++u) {
                if (u < nr) {
                    w[u] = __ldg(reinterpret_cast<const uint4*>(a.hidden + (rec_base + t0 + u) * a.row_stride) + c8);
                    if (F16) w[u] = f16x8_to_bf16x8(w[u]);
                    if (!RAW) { m[u] = a.mu[stat_base + t0 + u]; rs[u] = a.rstd[stat_base + t0 + u]; }
                }
            }
#pragma unroll
            for (int u = 0; u < 6; ++u) {
                if (u < nr) {
                    const float v[8] = {bf16_lo(w[u].x), bf16_hi(w[u].x), bf16_lo(w[u].y), bf16_hi(w[u].y),
                                        bf16_lo(w[u].z), bf16_hi(w[u].z), bf16_lo(w[u].w), bf16_hi(w[u].w)};
                    if (RAW) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) acc[k] += v[k];
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) acc[k] += (v[k] - m[u]) * rs[u];
                    }
                }
            }
        }
        if (kind == 1) {
            for (int t0 = s; t0 < e; t0 += 6) {
                const int nr = min(6, e - t0);
                uint4 x[6];
#pragma unroll
                for (int u = 0; u < 6; ++u) {
                    x[u] = make_uint4(0, 0, 0, 0);
                    if (u < nr) {
                        const int id = a.token_ids[rec_base + t0 + u];
                        if (id >= 0 && id < a.vocab)
                            x[u] = __ldg(reinterpret_cast<const uint4*>(a.lexical + int64_t(id) * H) + c8);
                        else if (c8 == 0)
                            atomicOr(a.flags, kFlagBounds);
                    }
                }
#pragma unroll
                for (int u = 0; u < 6; ++u) {
                    lex[0] += bf16_lo(x[u].x); lex[1] += bf16_hi(x[u].x);
                    lex[2] += bf16_lo(x[u].y); lex[3] += bf16_hi(x[u].y);
                    lex[4] += bf16_lo(x[u].z); lex[5] += bf16_hi(x[u].z);
                    lex[6] += bf16_lo(x[u].w); lex[7] += bf16_hi(x[u].w);
                }
            }
        }
        const int col = c8 * 8;
        if (RAW) {
            float* dst = kind == 0 ? a.q_sum + int64_t(idx) * H : (kind == 1 ? a.o_sum + int64_t(idx) * H : nullptr);
            if (dst) {
                reinterpret_cast<float4*>(dst + col)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                reinterpret_cast<float4*>(dst + col)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            if (kind == 1) {
                float* dx = a.x_sum + int64_t(idx) * H + col;
                reinterpret_cast<float4*>(dx)[0] = make_float4(lex[0], lex[1], lex[2], lex[3]);
                reinterpret_cast<float4*>(dx)[1] = make_float4(lex[4], lex[5], lex[6], lex[7]);
            }
            continue;
        }
        uint4 gw = __ldg(reinterpret_cast<const uint4*>(a.ln_w) + c8);
        uint4 bw = __ldg(reinterpret_cast<const uint4*>(a.ln_b) + c8);
        const float gam[8] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y),
                              bf16_lo(gw.z), bf16_hi(gw.z), bf16_lo(gw.w), bf16_hi(gw.w)};
        const float bet[8] = {bf16_lo(bw.x), bf16_hi(bw.x), bf16_lo(bw.y), bf16_hi(bw.y),
                              bf16_lo(bw.z), bf16_hi(bw.z), bf16_lo(bw.w), bf16_hi(bw.w)};
        float val[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) val[k] = acc[k] * inv_n * gam[k] + bet[k];
        uint4 vb;
        vb.x = pack_bf16(val[0], val[1]); vb.y = pack_bf16(val[2], val[3]);
        vb.z = pack_bf16(val[4], val[5]); vb.w = pack_bf16(val[6], val[7]);
        const float4 v0 = make_float4(val[0], val[1], val[2], val[3]);
        const float4 v1 = make_float4(val[4], val[5], val[6], val[7]);
        if (kind == 0) {
            float* u = a.u32 + int64_t(idx) * H + col;
            reinterpret_cast<float4*>(u)[0] = v0;
            reinterpret_cast<float4*>(u)[1] = v1;
            *reinterpret_cast<uint4*>(a.a_field + int64_t(idx) * a.ld_field + col) = vb;
            for (int j = a.q_opt_off[idx]; j < a.q_opt_off[idx + 1]; ++j)
                *reinterpret_cast<uint4*>(a.a_query + int64_t(j) * a.ld_query + 2 * H + col) = vb;
        } else if (kind == 1) {
            *reinterpret_cast<uint4*>(a.a_query + int64_t(idx) * a.ld_query + col) = vb;
            if (a.dbg_c) {
                reinterpret_cast<float4*>(a.dbg_c + int64_t(idx) * H + col)[0] = v0;
                reinterpret_cast<float4*>(a.dbg_c + int64_t(idx) * H + col)[1] = v1;
            }
            float xv[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) xv[k] = lex[k] * inv_n;
            float* x = a.x32 + int64_t(idx) * H + col;
            reinterpret_cast<float4*>(x)[0] = make_float4(xv[0], xv[1], xv[2], xv[3]);
            reinterpret_cast<float4*>(x)[1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
            uint4 xb;
            xb.x = pack_bf16(xv[0], xv[1]); xb.y = pack_bf16(xv[2], xv[3]);
            xb.z = pack_bf16(xv[4], xv[5]); xb.w = pack_bf16(xv[6], xv[7]);
            *reinterpret_cast<uint4*>(a.a_query + int64_t(idx) * a.ld_query + H + col) = xb;
        } else {
            float* g = a.g32 + int64_t(idx) * H + col;
            reinterpret_cast<float4*>(g)[0] = v0;
            reinterpret_cast<float4*>(g)[1] = v1;
            for (int q = a.rec_q_off[b]; q < a.rec_q_off[b + 1]; ++q)
                *reinterpret_cast<uint4*>(a.a_field + int64_t(q) * a.ld_field + H + col) = vb;
        }
    }
}

// =====================================================================
// A residual-stream projection finished and normalised in one pass: the projection's
// split-K partial products (S fp32 slabs from the tensor-core GEMM) are summed, then
// its bias, the type-embedding row (field projection) and the stream's previous value
// (residual projections) are added, the stream is updated, and the LayerNorm that
// follows the projection in the layer is applied (pre-LN of the next sub-layer, or the
// final option / field norm).
// One CTA of kAccGroups x 128 threads per row.  Group g sums slabs g, g + G, g + 2G, ...
// in that order (G = min(S, kAccGroups) groups, so that G slab loads are in flight per
// chunk); the group sums are then added in group order, so the result does not depend
// on timing.  Thread t of group 0 owns the 8-column chunks t, t + 128, ... for the rest.
// =====================================================================
constexpr int kAccGroups = 2;

template <int NCK>
__global__ void __launch_bounds__(128 * kAccGroups) layer_norm_acc_kernel(const LnAccArgs a) {
    griddep_wait();
    griddep_launch();
    __shared__ float4 xch[kAccGroups - 1][NCK][128][2];
    __shared__ float red[2][kAccGroups * 4];
    const int r = blockIdx.x, t = threadIdx.x & 127, grp = threadIdx.x >> 7;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D, nc = D >> 3;
    const int G = min(a.S, kAccGroups);
    float v[NCK][8];
#pragma unroll
    for (int k = 0; k < NCK; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) v[k][j] = 0.f;
    // group 0 requests everything else the row needs together with its slabs: bias,
    // type-embedding row, previous stream value and the LayerNorm affine
    uint4 bias_v[NCK], tab_v[NCK], lnw_v[NCK], lnb_v[NCK];
    float4 x_v[NCK][2];
    if (grp == 0) {
        const uint16_t* trow = a.row_table ? a.row_table + int64_t(a.row_idx[r]) * a.ld_table : nullptr;
#pragma unroll
        for (int k = 0; k < NCK; ++k) {
            const int c = t + 128 * k;
            if (c >= nc) continue;
            bias_v[k] = a.bias ? __ldg(reinterpret_cast<const uint4*>(a.bias) + c) : make_uint4(0, 0, 0, 0);
            tab_v[k] = trow ? __ldg(reinterpret_cast<const uint4*>(trow) + c) : make_uint4(0, 0, 0, 0);
            lnw_v[k] = __ldg(reinterpret_cast<const uint4*>(a.ln_w) + c);
            lnb_v[k] = __ldg(reinterpret_cast<const uint4*>(a.ln_b) + c);
            const float4* xr = reinterpret_cast<const float4*>(a.x + int64_t(r) * D) + 2 * c;
            x_v[k][0] = a.resid ? xr[0] : make_float4(0.f, 0.f, 0.f, 0.f);
            x_v[k][1] = a.resid ? xr[1] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (grp < G) {
#pragma unroll
        for (int k = 0; k < NCK; ++k) {
            const int c = t + 128 * k;
            if (c >= nc) continue;
            const float* pr = a.part + int64_t(r) * D + 8 * c;
#pragma unroll 4
            for (int sp = grp; sp < a.S; sp += G) {
                const float4 p0 = reinterpret_cast<const float4*>(pr + sp * a.part_stride)[0];
                const float4 p1 = reinterpret_cast<const float4*>(pr + sp * a.part_stride)[1];
                v[k][0] += p0.x; v[k][1] += p0.y; v[k][2] += p0.z; v[k][3] += p0.w;
                v[k][4] += p1.x; v[k][5] += p1.y; v[k][6] += p1.z; v[k][7] += p1.w;
            }
            if (grp > 0) {
                xch[grp - 1][k][t][0] = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
                xch[grp - 1][k][t][1] = make_float4(v[k][4], v[k][5], v[k][6], v[k][7]);
            }
        }
    }
    __syncthreads();
    float s = 0.f;
    if (grp == 0) {
#pragma unroll
        for (int k = 0; k < NCK; ++k) {
            const int c = t + 128 * k;
            if (c >= nc) continue;
            for (int g = 1; g < G; ++g) {
                const float4 p0 = xch[g - 1][k][t][0], p1 = xch[g - 1][k][t][1];
                v[k][0] += p0.x; v[k][1] += p0.y; v[k][2] += p0.z; v[k][3] += p0.w;
                v[k][4] += p1.x; v[k][5] += p1.y; v[k][6] += p1.z; v[k][7] += p1.w;
            }
            if (a.bias) {
                const uint4 b = bias_v[k];
                v[k][0] += bf16_lo(b.x); v[k][1] += bf16_hi(b.x); v[k][2] += bf16_lo(b.y); v[k][3] += bf16_hi(b.y);
                v[k][4] += bf16_lo(b.z); v[k][5] += bf16_hi(b.z); v[k][6] += bf16_lo(b.w); v[k][7] += bf16_hi(b.w);
            }
            if (a.row_table) {
                const uint4 b = tab_v[k];
                v[k][0] += bf16_lo(b.x); v[k][1] += bf16_hi(b.x); v[k][2] += bf16_lo(b.y); v[k][3] += bf16_hi(b.y);
                v[k][4] += bf16_lo(b.z); v[k][5] += bf16_hi(b.z); v[k][6] += bf16_lo(b.w); v[k][7] += bf16_hi(b.w);
            }
            float4* xr = reinterpret_cast<float4*>(a.x + int64_t(r) * D) + 2 * c;
            if (a.resid) {
                const float4 o0 = x_v[k][0], o1 = x_v[k][1];
                v[k][0] += o0.x; v[k][1] += o0.y; v[k][2] += o0.z; v[k][3] += o0.w;
                v[k][4] += o1.x; v[k][5] += o1.y; v[k][6] += o1.z; v[k][7] += o1.w;
            }
            xr[0] = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
            xr[1] = make_float4(v[k][4], v[k][5], v[k][6], v[k][7]);
#pragma unroll
            for (int j = 0; j < 8; ++j) s += v[k][j];
        }
    }
    s = warp_sum(s);
    if (lane == 0) red[0][warp] = s;
    __syncthreads();
    const float m = (red[0][0] + red[0][1] + red[0][2] + red[0][3]) / float(D);
    float q = 0.f;
    if (grp == 0) {
#pragma unroll
        for (int k = 0; k < NCK; ++k) {
            if (t + 128 * k < nc) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float d = v[k][j] - m;
                    q += d * d;
                }
            }
        }
    }
    q = warp_sum(q);
    if (lane == 0) red[1][warp] = q;
    __syncthreads();
    if (grp != 0) return;
    const float rs = rsqrtf((red[1][0] + red[1][1] + red[1][2] + red[1][3]) / float(D) + 1e-5f);
#pragma unroll
    for (int k = 0; k < NCK; ++k) {
        const int c = t + 128 * k;
        if (c >= nc) continue;
        const uint4 wv = lnw_v[k], bv = lnb_v[k];
        const float gm[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                             bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
        const float bt[8] = {bf16_lo(bv.x), bf16_hi(bv.x), bf16_lo(bv.y), bf16_hi(bv.y),
                             bf16_lo(bv.z), bf16_hi(bv.z), bf16_lo(bv.w), bf16_hi(bv.w)};
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = (v[k][j] - m) * rs * gm[j] + bt[j];
        if (a.out_bf16) {
            uint4 o;
            o.x = pack_bf16(y[0], y[1]); o.y = pack_bf16(y[2], y[3]);
            o.z = pack_bf16(y[4], y[5]); o.w = pack_bf16(y[6], y[7]);
            reinterpret_cast<uint4*>(a.out_bf16 + int64_t(r) * D)[c] = o;
        }
        if (a.out_f32) {
            float4* o = reinterpret_cast<float4*>(a.out_f32 + int64_t(r) * D);
            o[2 * c] = make_float4(y[0], y[1], y[2], y[3]);
            o[2 * c + 1] = make_float4(y[4], y[5], y[6], y[7]);
        }
        if (a.z) {  // the scorer MLP input of every option of this row's question
            const int j0 = a.z_opt_off[r], j1 = a.z_opt_off[r + 1];
            for (int jb = j0; jb < j1; jb += 4) {
                float4 ov[4][2];
#pragma unroll
                for (int u = 0; u < 4; ++u)  // four options' chunks requested before any is used
                    if (jb + u < j1) {
                        const float4* op = reinterpret_cast<const float4*>(a.z_o_hat + int64_t(jb + u) * D) + 2 * c;
                        ov[u][0] = op[0];
                        ov[u][1] = op[1];
                    }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (jb + u >= j1) break;
                    const float o[8] = {ov[u][0].x, ov[u][0].y, ov[u][0].z, ov[u][0].w,
                                        ov[u][1].x, ov[u][1].y, ov[u][1].z, ov[u][1].w};
                    uint4 pf, po, pm, pd;
                    pf.x = pack_bf16(y[0], y[1]); pf.y = pack_bf16(y[2], y[3]);
                    pf.z = pack_bf16(y[4], y[5]); pf.w = pack_bf16(y[6], y[7]);
                    po.x = pack_bf16(o[0], o[1]); po.y = pack_bf16(o[2], o[3]);
                    po.z = pack_bf16(o[4], o[5]); po.w = pack_bf16(o[6], o[7]);
                    pm.x = pack_bf16(y[0] * o[0], y[1] * o[1]); pm.y = pack_bf16(y[2] * o[2], y[3] * o[3]);
                    pm.z = pack_bf16(y[4] * o[4], y[5] * o[5]); pm.w = pack_bf16(y[6] * o[6], y[7] * o[7]);
                    pd.x = pack_bf16(fabsf(y[0] - o[0]), fabsf(y[1] - o[1]));
                    pd.y = pack_bf16(fabsf(y[2] - o[2]), fabsf(y[3] - o[3]));
                    pd.z = pack_bf16(fabsf(y[4] - o[4]), fabsf(y[5] - o[5]));
                    pd.w = pack_bf16(fabsf(y[6] - o[6]), fabsf(y[7] - o[7]));
                    uint4* zr = reinterpret_cast<uint4*>(a.z + int64_t(jb + u) * 4 * D);
                    zr[c] = pf;
                    zr[(D >> 3) + c] = po;
                    zr[2 * (D >> 3) + c] = pm;
                    zr[3 * (D >> 3) + c] = pd;
                }
            }
        }
    }
}

// =====================================================================
// Field aggregation, summary part ("clef-4bit JointSchemaHead walkthrough" section 3
// step 3, option-weighted summary): alpha = softmax_j(w_a . o_hat_j + b_a) over
// the question's options; summary = sum_j alpha_j o_hat_j, written as bf16 into
// the field projection's input row.  One CTA per question.
// =====================================================================
__global__ void __launch_bounds__(256) field_pool_kernel(const float* __restrict__ o_hat, int D,
                                                        const int32_t* __restrict__ q_opt_off,
                                                        const uint16_t* __restrict__ w_a, const uint16_t* __restrict__ b_a,
                                                        uint16_t* __restrict__ out, int64_t ldo, int col_off) {
    griddep_wait();
    griddep_launch();
    __shared__ float sc[256];
    const int q = blockIdx.x;
    const int j0 = q_opt_off[q], n = q_opt_off[q + 1] - j0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < n; j += 8) {
        const float4* row = reinterpret_cast<const float4*>(o_hat + int64_t(j0 + j) * D);
        const uint2* w2 = reinterpret_cast<const uint2*>(w_a);
        float s = 0.f;
#pragma unroll 8
        for (int c = lane; c < D / 4; c += 32) {
            const float4 x = row[c];
            const uint2 w = w2[c];
            s += x.x * bf16_lo(w.x) + x.y * bf16_hi(w.x) + x.z * bf16_lo(w.y) + x.w * bf16_hi(w.y);
        }
        s = warp_sum(s);
        if (lane == 0) sc[j] = s + bf16_to_float(b_a[0]);
    }
    __syncthreads();
    if (warp == 0) {
        float m = -INFINITY;
        for (int j = lane; j < n; j += 32) m = fmaxf(m, sc[j]);
        m = warp_max(m);
        float z = 0.f;
        for (int j = lane; j < n; j += 32) z += expf(sc[j] - m);
        z = warp_sum(z);
        __syncwarp();
        for (int j = lane; j < n; j += 32) sc[j] = expf(sc[j] - m) / z;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < D / 4; c += blockDim.x) {  // 4 columns per thread
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int j = 0; j < n; ++j) {
            const float a = sc[j];
            const float4 x = reinterpret_cast<const float4*>(o_hat + int64_t(j0 + j) * D)[c];
            acc.x += a * x.x; acc.y += a * x.y; acc.z += a * x.z; acc.w += a * x.w;
        }
        *reinterpret_cast<uint2*>(out + int64_t(q) * ldo + col_off + 4 * c) =
            make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
    }
}

// =====================================================================
// Self-attention among one record's fields (joint layers, "clef-4bit JointSchemaHead
// walkthrough" section 3 step 3: fields are mutually visible).  One CTA per
// (record, head); fp32 scores and softmax; at most kMaxFields fields per record.
// qkv is bf16 [Q][3D] (q | k | v), out bf16 [Q][D].
// =====================================================================
__global__ void __launch_bounds__(128) field_attn_kernel(const uint16_t* __restrict__ qkv, int D,
                                                        const int32_t* __restrict__ rec_q_off, float scale,
                                                        uint16_t* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    __shared__ float sq[kMaxFields][65], sk[kMaxFields][65], sv[kMaxFields][65];
    __shared__ float sp[kMaxFields][kMaxFields + 1];
    const int b = blockIdx.x, h = blockIdx.y;
    const int q0 = rec_q_off[b], n = rec_q_off[b + 1] - q0;
    // 16-byte loads: thread i takes columns 8 (i % 8) .. + 7 of field i / 8 of q, k and v
    for (int i = threadIdx.x; i < n * 8; i += blockDim.x) {
        const int r = i >> 3, c8 = (i & 7) * 8;
        const uint16_t* row = qkv + int64_t(q0 + r) * 3 * D + h * 64 + c8;
        const uint4 a = *reinterpret_cast<const uint4*>(row);
        const uint4 bk = *reinterpret_cast<const uint4*>(row + D);
        const uint4 bv = *reinterpret_cast<const uint4*>(row + 2 * D);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wk[4] = {bk.x, bk.y, bk.z, bk.w}, wv[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sq[r][c8 + 2 * j] = bf16_lo(wa[j]); sq[r][c8 + 2 * j + 1] = bf16_hi(wa[j]);
            sk[r][c8 + 2 * j] = bf16_lo(wk[j]); sk[r][c8 + 2 * j + 1] = bf16_hi(wk[j]);
            sv[r][c8 + 2 * j] = bf16_lo(wv[j]); sv[r][c8 + 2 * j + 1] = bf16_hi(wv[j]);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n * n; i += blockDim.x) {
        const int r = i / n, c = i % n;
        float s = 0.f;
#pragma unroll 8
        for (int d = 0; d < 64; ++d) s += sq[r][d] * sk[c][d];
        sp[r][c] = s * scale;
    }
    __syncthreads();
    if (threadIdx.x < n) {
        const int r = threadIdx.x;
        float m = -INFINITY;
        for (int c = 0; c < n; ++c) m = fmaxf(m, sp[r][c]);
        float z = 0.f;
        for (int c = 0; c < n; ++c) { const float e = expf(sp[r][c] - m); sp[r][c] = e; z += e; }
        const float inv = 1.f / z;
        for (int c = 0; c < n; ++c) sp[r][c] *= inv;
    }
    __syncthreads();
    // thread i writes columns 8 (i % 8) .. + 7 of field i / 8 with one 16-byte store
    for (int i = threadIdx.x; i < n * 8; i += blockDim.x) {
        const int r = i >> 3, c8 = (i & 7) * 8;
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int c = 0; c < n; ++c) {
            const float p = sp[r][c];
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] += p * sv[c][c8 + j];
        }
        uint4 w;
        w.x = pack_bf16(o[0], o[1]); w.y = pack_bf16(o[2], o[3]);
        w.z = pack_bf16(o[4], o[5]); w.w = pack_bf16(o[6], o[7]);
        *reinterpret_cast<uint4*>(out + int64_t(q0 + r) * D + h * 64 + c8) = w;
    }
}

// =====================================================================
// Scoring and per-question softmax, one CTA per question
// ("clef-4bit JointSchemaHead walkthrough" section 3 step 4;
// "clef-flash-CoreAI metadata.json" decision.softmax and decision.response):
//   logit_j = cos(x_j, u_q + g_b) + sigmoid(gate) * (joint_scale * cos(f_hat_q, o_hat_j) + mlp_j)
//   mlp_j   = w2 . hidden_j + b2  (hidden_j = GELU(W1 z_j + b1) from the GEMM)
//   p = softmax over the question's options; answers by question type.
// =====================================================================
__global__ void __launch_bounds__(256) score_softmax_kernel(ScoreArgs a) {
    griddep_wait();
    griddep_launch();
    extern __shared__ float4 s_dyn4[];  // u_q + g_b [H], then f_hat_q [D]: read once, used by every option
    __shared__ float s_logit[256];
    __shared__ float s_red[8];
    __shared__ float s_anchor_norm;
    const int q = blockIdx.x;
    const int b = a.q_rec[q];
    const int j0 = a.q_opt_off[q], n = a.q_opt_off[q + 1] - j0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, D = a.D;
    const float4* u4 = reinterpret_cast<const float4*>(a.u32 + int64_t(q) * H);
    const float4* g4 = reinterpret_cast<const float4*>(a.g32 + int64_t(b) * H);
    const float4* f4 = reinterpret_cast<const float4*>(a.f_hat + int64_t(q) * D);
    float4* s_ug = s_dyn4;
    float4* s_f = s_dyn4 + H / 4;
    // anchor u_q + g_b and its norm
    float ss = 0.f;
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
        const float4 uv = u4[c], gv = g4[c];
        const float4 v = make_float4(uv.x + gv.x, uv.y + gv.y, uv.z + gv.z, uv.w + gv.w);
        s_ug[c] = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    for (int c = threadIdx.x; c < D / 4; c += blockDim.x) s_f[c] = f4[c];
    ss = warp_sum(ss);
    if (lane == 0) s_red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += s_red[w];
        s_anchor_norm = fmaxf(sqrtf(t), 1e-8f);
    }
    __syncthreads();
    const float gate = 1.0f / (1.0f + expf(-bf16_to_float(a.gate[0])));
    const float jscale = bf16_to_float(a.joint_scale[0]);
    for (int jj = warp; jj < n; jj += 8) {
        const int j = j0 + jj;
        const float4* x4 = reinterpret_cast<const float4*>(a.x32 + int64_t(j) * H);
        float xa = 0.f, xx = 0.f;
#pragma unroll 8
        for (int c = lane; c < H / 4; c += 32) {
            const float4 xv = x4[c], av = s_ug[c];
            xa += xv.x * av.x + xv.y * av.y + xv.z * av.z + xv.w * av.w;
            xx += xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
        }
        const float4* o4 = reinterpret_cast<const float4*>(a.o_hat + int64_t(j) * D);
        const uint2* hm = reinterpret_cast<const uint2*>(a.mlp_hidden + int64_t(j) * D);
        const uint2* w2 = reinterpret_cast<const uint2*>(a.w2);
        float fo = 0.f, ff = 0.f, oo = 0.f, mm = 0.f;
#pragma unroll 8
        for (int c = lane; c < D / 4; c += 32) {
            const float4 fv = s_f[c], ov = o4[c];
            fo += fv.x * ov.x + fv.y * ov.y + fv.z * ov.z + fv.w * ov.w;
            ff += fv.x * fv.x + fv.y * fv.y + fv.z * fv.z + fv.w * fv.w;
            oo += ov.x * ov.x + ov.y * ov.y + ov.z * ov.z + ov.w * ov.w;
            const uint2 hv = hm[c], wv = w2[c];
            mm += bf16_lo(hv.x) * bf16_lo(wv.x) + bf16_hi(hv.x) * bf16_hi(wv.x) + bf16_lo(hv.y) * bf16_lo(wv.y) +
                  bf16_hi(hv.y) * bf16_hi(wv.y);
        }
        xa = warp_sum(xa); xx = warp_sum(xx); fo = warp_sum(fo); ff = warp_sum(ff); oo = warp_sum(oo); mm = warp_sum(mm);
        if (lane == 0) {
            const float prior = xa / (fmaxf(sqrtf(xx), 1e-8f) * s_anchor_norm);
            const float joint = fo / (fmaxf(sqrtf(ff), 1e-8f) * fmaxf(sqrtf(oo), 1e-8f));
            const float mlp = mm + bf16_to_float(a.b2[0]);
            s_logit[jj] = prior + gate * (jscale * joint + mlp);
        }
    }
    __syncthreads();
    if (warp == 0) {
        float m = -INFINITY;
        for (int j = lane; j < n; j += 32) m = fmaxf(m, s_logit[j]);
        m = warp_max(m);
        float z = 0.f;
        for (int j = lane; j < n; j += 32) z += expf(s_logit[j] - m);
        z = warp_sum(z);
        float ev = 0.f;
        for (int j = lane; j < n; j += 32) {
            const float p = expf(s_logit[j] - m) / z;
            a.logits[j0 + j] = s_logit[j];
            a.probs[j0 + j] = p;
            ev += float(j) * p;
        }
        ev = warp_sum(ev);
        if (lane == 0) {
            // first maximum in option order (ties -> lowest index)
            int k = 0;
            for (int j = 1; j < n; ++j)
                if (s_logit[j] > s_logit[k]) k = j;
            const float pk = expf(s_logit[k] - m) / z;
            const int t = a.q_type[q];
            a.q_argmax[q] = k;
            a.q_conf[q] = pk;
            a.q_value[q] = t == 0 ? expf(s_logit[0] - m) / z : (t == 1 ? pk : ev);
        }
    }
}

// =====================================================================
// Weight preparation.
// Memory K/V projections with the memory LayerNorm folded in: for weight row n,
//   W'[n][k] = bf16(W[n][k] * gamma[k]),  c[n] = sum_k W'[n][k],
//   b'[n] = sum_k beta[k] * W[n][k] + bias[n]
// so that W LN(h) + bias = rstd * (W' h - mu c) + b'.
// =====================================================================
__global__ void __launch_bounds__(256) fold_kv_kernel(FoldArgs a) {
    __shared__ float red[2][8];
    const int n = blockIdx.x;
    const int mat = n / a.D, r = n % a.D;
    const uint16_t* W = a.w[mat] + int64_t(r) * a.H;
    uint16_t* Wp = a.out_w + int64_t(n) * a.H;
    float cs = 0.f, bs = 0.f;
    for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
        const float w = bf16_to_float(W[k]);
        const uint16_t wp = float_to_bf16(w * bf16_to_float(a.gamma[k]));
        Wp[k] = wp;
        cs += bf16_to_float(wp);
        bs += w * bf16_to_float(a.beta[k]);
    }
    cs = warp_sum(cs);
    bs = warp_sum(bs);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { red[0][warp] = cs; red[1][warp] = bs; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float c = 0.f, bb = 0.f;
        for (int w = 0; w < 8; ++w) { c += red[0][w]; bb += red[1][w]; }
        a.out_c[n] = c;
        a.out_b[n] = bb + bf16_to_float(a.bias[mat][r]);
    }
}

// Launch-plan upload: the host's plan tables travel as kernel parameters (copied by
// the launch itself, so no host buffer has to outlive the call and nothing waits).
struct alignas(16) PlanChunk {
    int32_t data[kPlanChunkInts];  // first: 16-byte aligned for vector reads
    int32_t n;
};
static_assert(kPlanChunkInts % 4 == 0, "plan chunks start on 16-byte boundaries of the destination");
static_assert(sizeof(PlanChunk) + sizeof(int32_t*) <= 32764, "kernel parameters are limited to 32,764 bytes");

// One 16-byte unit per thread over several CTAs (reads of the parameter block by
// different lanes do not broadcast, so the copy is spread out); dst is 16-byte aligned.
// The launch also clears up to two 16-byte-aligned regions (z0: n0 units, z1: n1 units).
__global__ void __launch_bounds__(256) plan_upload_kernel(int32_t* __restrict__ dst, const __grid_constant__ PlanChunk c,
                                                         int4* __restrict__ z0, int n0, int4* __restrict__ z1,
                                                         int n1) {
    griddep_wait();
    griddep_launch();
    const int i = int(blockIdx.x * blockDim.x + threadIdx.x);
    const int n4 = c.n >> 2;
    if (i < n4) reinterpret_cast<int4*>(dst)[i] = reinterpret_cast<const int4*>(c.data)[i];
    if (i < (c.n & 3)) dst[4 * n4 + i] = c.data[4 * n4 + i];
    for (int k = i; k < n0 + n1; k += int(gridDim.x * blockDim.x)) {
        if (k < n0) z0[k] = make_int4(0, 0, 0, 0);
        else z1[k - n0] = make_int4(0, 0, 0, 0);
    }
}

// dst[r][col_off + c] = src[r][c] for a [rows][cols] bf16 block (16-byte units).
__global__ void __launch_bounds__(256) copy_cols_kernel(uint16_t* __restrict__ dst, int64_t ld_dst, int col_off,
                                                       const uint16_t* __restrict__ src, int64_t ld_src, int rows,
                                                       int cols) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int c8 = cols >> 3;
    if (i >= int64_t(rows) * c8) return;
    const int r = int(i / c8), c = int(i % c8) * 8;
    *reinterpret_cast<uint4*>(dst + int64_t(r) * ld_dst + col_off + c) =
        *reinterpret_cast<const uint4*>(src + int64_t(r) * ld_src + c);
}

// =====================================================================
// Self-test of the bounded waits: one thread waits on an mbarrier that nothing ever
// completes, then on a global flag that nothing sets, each with a short limit, so each
// wait runs out, sets the timeout bit of the status word and returns; flags[2] records
// which waits gave up (bit 0: barrier, bit 1: flag).  No thread hangs and nothing faults.
// =====================================================================
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(int* flags, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        int gave_up = 0;
        if (!mbar_wait_bounded(&bar, 0, nullptr, flags, limit_ns)) gave_up |= 1;  // phase 0 never completes
        // the flag at byte 128 of the cleared block stays 0; the wait is for 1
        if (!flag_wait_bounded(reinterpret_cast<const uint64_t*>(flags + 32), 1, nullptr, flags, limit_ns))
            gave_up |= 2;
        flags[2] = gave_up;
    }
    __syncwarp();
}

// ----------------------------------------------------------------- launchers

cudaError_t launch_wait_timeout_selftest(int* flags, uint64_t limit_ns, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(flags, limit_ns);
    return counted(cudaGetLastError());
}

cudaError_t launch_zero_slack(uint16_t* kv, int ldkv, const int32_t* rec_row_off, const int32_t* lengths, int B,
                              cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    return launch_pdl(zero_slack_kernel, dim3(B), dim3(256), 0, s, kv, ldkv, rec_row_off, lengths);
}

cudaError_t launch_span_pool(const SpanPoolArgs& a, int n_items, bool raw, cudaStream_t s) {
    if (n_items <= 0) return cudaSuccess;
    if (a.in_f16) {
        if (raw) return launch_pdl(span_pool_kernel<true, true>, dim3(n_items), dim3(256), 0, s, a);
        return launch_pdl(span_pool_kernel<false, true>, dim3(n_items), dim3(256), 0, s, a);
    }
    if (raw) return launch_pdl(span_pool_kernel<true, false>, dim3(n_items), dim3(256), 0, s, a);
    return launch_pdl(span_pool_kernel<false, false>, dim3(n_items), dim3(256), 0, s, a);
}

cudaError_t launch_f16_rows_to_bf16(const uint16_t* src, int64_t ld_src, int rows, int H, uint16_t* dst,
                                    cudaStream_t s) {
    const int64_t n = int64_t(rows) * (H / 8);
    if (n <= 0) return cudaSuccess;
    return launch_pdl(f16_rows_to_bf16_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, s, src, ld_src, rows,
                      H, dst);
}

cudaError_t launch_layer_norm_acc(const LnAccArgs& a, cudaStream_t s) {
    if (a.rows <= 0) return cudaSuccess;
    if (a.D % 8 != 0 || a.D > 2048 || a.S < 1 || !a.part || !a.x || !a.ln_w || !a.ln_b) return cudaErrorInvalidValue;
    const dim3 block(128 * kAccGroups);
    if (a.D <= 1024) return launch_pdl(layer_norm_acc_kernel<1>, dim3(unsigned(a.rows)), block, 0, s, a);
    return launch_pdl(layer_norm_acc_kernel<2>, dim3(unsigned(a.rows)), block, 0, s, a);
}

cudaError_t launch_field_pool(const float* o_hat, int D, const int32_t* q_opt_off, int Q, const uint16_t* w_a,
                              const uint16_t* b_a, uint16_t* out, int64_t ldo, int col_off, cudaStream_t s) {
    if (Q <= 0) return cudaSuccess;
    return launch_pdl(field_pool_kernel, dim3(Q), dim3(256), 0, s, o_hat, D, q_opt_off, w_a, b_a, out, ldo, col_off);
}

cudaError_t launch_field_attn(const uint16_t* qkv, int D, int heads, const int32_t* rec_q_off, int B, float scale,
                              uint16_t* out, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    return launch_pdl(field_attn_kernel, dim3(B, heads), dim3(128), 0, s, qkv, D, rec_q_off, scale, out);
}

cudaError_t launch_score_softmax(const ScoreArgs& a, int Q, cudaStream_t s) {
    if (Q <= 0) return cudaSuccess;
    const size_t smem = size_t(a.H + a.D) * sizeof(float);  // at most 40 KB for supported widths
    return launch_pdl(score_softmax_kernel, dim3(Q), dim3(256), smem, s, a);
}

cudaError_t launch_plan_upload(int32_t* dst, const int32_t* src, size_t n, void* z0, size_t z0_bytes, void* z1,
                               size_t z1_bytes, cudaStream_t s) {
    if ((z0_bytes | z1_bytes) % 16 || (reinterpret_cast<uintptr_t>(z0) | reinterpret_cast<uintptr_t>(z1)) % 16 ||
        z0_bytes / 16 + z1_bytes / 16 >= (size_t(1) << 30))
        return cudaErrorInvalidValue;
    PlanChunk c;
    int n0 = int(z0_bytes / 16), n1 = int(z1_bytes / 16);  // cleared by the first chunk's launch
    for (size_t off = 0; off < n; off += kPlanChunkInts) {
        c.n = int32_t(n - off < size_t(kPlanChunkInts) ? n - off : size_t(kPlanChunkInts));
        for (int i = 0; i < c.n; ++i) c.data[i] = src[off + i];
        const int units = std::max((c.n + 3) / 4, std::min(n0 + n1, 64 * 1024));
        const unsigned grid = unsigned((units + 255) / 256);
        const cudaError_t e = launch_pdl(plan_upload_kernel, dim3(grid), dim3(256), 0, s, dst + off, c,
                                         static_cast<int4*>(z0), n0, static_cast<int4*>(z1), n1);
        if (e != cudaSuccess) return e;
        n0 = n1 = 0;
    }
    return cudaSuccess;
}

cudaError_t launch_fold_kv(const FoldArgs& a, int rows, cudaStream_t s) {
    fold_kv_kernel<<<rows, 256, 0, s>>>(a);
    return counted(cudaGetLastError());
}

cudaError_t launch_copy_cols(uint16_t* dst, int64_t ld_dst, int col_off, const uint16_t* src, int64_t ld_src,
                             int rows, int cols, cudaStream_t s) {
    const int64_t n = int64_t(rows) * (cols / 8);
    if (n <= 0) return cudaSuccess;
    copy_cols_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(dst, ld_dst, col_off, src, ld_src, rows, cols);
    return counted(cudaGetLastError());
}

}  // namespace clef
