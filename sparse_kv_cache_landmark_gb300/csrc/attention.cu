// GQA decode attention over the gathered sparse blocks plus the GPU-resident
// recent window, the two parts fused by log-sum-exp ("Scaling Attention Beyond
// GPUs for LLM Inference", abstract; DualDecoder core claim: attention over the
// miss-corrected buffer equals attention over the true sparse selection).
//
// Decode attention at r = Hq / Hkv <= 16 query rows is bound by the HBM read
// of K and V (about 4 flop per byte).  The kernel keeps the instruction count
// per token low with mma.sync m16n8k16 bf16 (the r query rows of a KV group
// fill the M = 16 rows; rows past r are zero) and loads K and V straight from
// global memory into fragment registers with 16-byte loads:
//  * S = Q K^T: the contraction over channels may use any channel order, as
//    long as Q and K use the same one.  Lane (g, t) loads 16 contiguous bytes
//    of key row g (channels 32s + 8t .. +8) and uses them as the B fragments
//    of k-steps 2s and 2s+1; the Q fragments are loaded with the same map.
//  * O += P V: lane (g, t) needs, for output column g of each n-tile, the
//    values of tokens 2t, 2t+1, 2t+8, 2t+9.  Output column g of n-tile j is
//    channel (d/8) g + j, so the lane loads d/8 contiguous channels of those 4
//    token rows and pairs tokens with byte permutes.
// Work: a work item is a run of 16-token tiles of one (request, KV head)
// group and one part (0 sparse, 1 window); a CTA's 4 warps keep online-softmax
// state over interleaved tiles of the item, merge in shared memory and write
// one unnormalised partial (m, l, acc).  The CTA finishing a group's last item
// (atomic ticket) merges the partials of each part and fuses the two parts.
// Two kernels share this math: the register-direct kernel (one CTA per item of
// up to ATT_TILES_PER_ITEM tiles; fragments loaded from global memory) and the
// TMA-staged persistent kernel (one balanced tile range per CTA; tiles copied
// into shared memory by bulk copies ahead of the math).
#include <math.h>

#include "kvo_internal.cuh"
#include "tma_ptx.cuh"

namespace kvo {

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2f(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void mma_bf16_16816(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1, float c0, float c1,
                                               float c2, float c3) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};\n"
        : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

constexpr float kLn2 = 0.69314718055994530942f;

// D: head dim (64|128).  NR: 1 -> query rows 0..7 (r <= 8), 2 -> rows 0..15.
#ifndef KVO_ATT_PREFETCH
#define KVO_ATT_PREFETCH 1   // prefetch each warp's next tile into L2
#endif
#ifndef KVO_ATT_MINB_NR1
#define KVO_ATT_MINB_NR1 4   // resident CTAs per SM requested for r <= 8 (caps registers at 128)
#endif

// One warp's online-softmax state over 16-token tiles, and the tile math shared
// by both attention kernels.  Lane (g, t): K fragments are 16-byte chunks of key
// rows g and 8+g at channels 32s + 8t; V fragments are d/8 channels (d/8)g ..
// of value rows 2t, 2t+1, 2t+8, 2t+9 of the tile.
template <int D, int NR>
struct WarpAttn {
    static constexpr int KS = D / 16, CH = D / 32, NT = D / 8, CPT = D / 8;
    uint32_t qa0[KS], qa1[KS], qa2[KS], qa3[KS];
    float acc[NT][2 * NR];   // NR == 1: only rows 0..7 exist, so only c0/c1 are kept
    float m0, m1, l0, l1;

    // the lane's Q words: rows g (w0) and 8+g (w1), channels 32s + 8t .. +8
    static __device__ __forceinline__ void load_q(const uint16_t* q0, const uint16_t* q1, bool v0, bool v1, int tq,
                                                  uint4 (&w0)[CH], uint4 (&w1)[CH]) {
#pragma unroll
        for (int s = 0; s < CH; ++s) {
            w0[s] = v0 ? ldg16(q0 + 32 * s + 8 * tq) : make_uint4(0u, 0u, 0u, 0u);
            w1[s] = (NR == 2 && v1) ? ldg16(q1 + 32 * s + 8 * tq) : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    __device__ __forceinline__ void init(const uint16_t* q0, const uint16_t* q1, bool v0, bool v1, int tq) {
        uint4 w0[CH], w1[CH];
        load_q(q0, q1, v0, v1, tq, w0, w1);
        init_from(w0, w1);
    }

    __device__ __forceinline__ void init_from(const uint4 (&w0)[CH], const uint4 (&w1)[CH]) {
#pragma unroll
        for (int s = 0; s < CH; ++s) {
            qa0[2 * s] = w0[s].x; qa2[2 * s] = w0[s].y; qa0[2 * s + 1] = w0[s].z; qa2[2 * s + 1] = w0[s].w;
            qa1[2 * s] = w1[s].x; qa3[2 * s] = w1[s].y; qa1[2 * s + 1] = w1[s].z; qa3[2 * s + 1] = w1[s].w;
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2 * NR; ++e) acc[j][e] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    // S = Q K^T for the 16 tokens of a tile (two n8 tiles)
    __device__ __forceinline__ void qk(const uint4 (&kf)[2][CH], float (&s)[2][4]) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint4 w = kf[nt][ks >> 1];
                const uint32_t b0 = (ks & 1) ? w.z : w.x;
                const uint32_t b1 = (ks & 1) ? w.w : w.y;
                if constexpr (NR == 2) {
                    mma_bf16_16816(s[nt][0], s[nt][1], s[nt][2], s[nt][3], qa0[ks], qa1[ks], qa2[ks], qa3[ks], b0,
                                   b1, s[nt][0], s[nt][1], s[nt][2], s[nt][3]);
                } else {
                    float d2, d3;
                    mma_bf16_16816(s[nt][0], s[nt][1], d2, d3, qa0[ks], 0u, qa2[ks], 0u, b0, b1, s[nt][0], s[nt][1],
                                   0.f, 0.f);
                }
            }
        }
    }

    // online softmax of tokens tb .. tb+15 (valid below n_tok), log2 domain;
    // gives the bf16 P fragments and the rescale factors of the old state
    __device__ __forceinline__ void softmax(const float (&s)[2][4], int tb, int n_tok, float scale_log2, int tq,
                                            uint32_t (&pa)[4], float& al0, float& al1) {
        // lane holds tokens 2t, 2t+1 of each n8 tile
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t0 = tb + 8 * nt + 2 * tq;
#pragma unroll
            for (int e = 0; e < 4; ++e) x[nt][e] = (t0 + (e & 1) < n_tok) ? s[nt][e] * scale_log2 : -INFINITY;
        }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        const float mn0 = fmaxf(m0, mx0);
        al0 = ex2f(m0 - mn0);
        m0 = mn0;
        float p[2][4];
        p[0][0] = ex2f(x[0][0] - mn0); p[0][1] = ex2f(x[0][1] - mn0);
        p[1][0] = ex2f(x[1][0] - mn0); p[1][1] = ex2f(x[1][1] - mn0);
        l0 = l0 * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        al1 = 1.f;
        if (NR == 2) {
            float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn1 = fmaxf(m1, mx1);
            al1 = ex2f(m1 - mn1);
            m1 = mn1;
            p[0][2] = ex2f(x[0][2] - mn1); p[0][3] = ex2f(x[0][3] - mn1);
            p[1][2] = ex2f(x[1][2] - mn1); p[1][3] = ex2f(x[1][3] - mn1);
            l1 = l1 * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
        } else {
            p[0][2] = p[0][3] = p[1][2] = p[1][3] = 0.f;
        }
        pa[0] = pack_bf16(p[0][0], p[0][1]);
        pa[1] = pack_bf16(p[0][2], p[0][3]);
        pa[2] = pack_bf16(p[1][0], p[1][1]);
        pa[3] = pack_bf16(p[1][2], p[1][3]);
    }

    // O = O * alpha + P V
    __device__ __forceinline__ void pv(const uint4 (&vf)[4][CPT / 8], const uint32_t (&pa)[4], float al0, float al1) {
        const uint32_t pa0 = pa[0], pa1 = pa[1], pa2 = pa[2], pa3 = pa[3];
#pragma unroll
        for (int c = 0; c < CPT / 8; ++c) {
            const uint32_t va[4] = {vf[0][c].x, vf[0][c].y, vf[0][c].z, vf[0][c].w};
            const uint32_t vb[4] = {vf[1][c].x, vf[1][c].y, vf[1][c].z, vf[1][c].w};
            const uint32_t vc[4] = {vf[2][c].x, vf[2][c].y, vf[2][c].z, vf[2][c].w};
            const uint32_t vd[4] = {vf[3][c].x, vf[3][c].y, vf[3][c].z, vf[3][c].w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    const int j = 8 * c + 2 * w + hi;   // n-tile == channel offset within the lane's CPT
                    const uint32_t sel = hi ? 0x7632u : 0x5410u;
                    const uint32_t b0 = __byte_perm(va[w], vb[w], sel);
                    const uint32_t b1 = __byte_perm(vc[w], vd[w], sel);
                    if constexpr (NR == 2) {
                        mma_bf16_16816(acc[j][0], acc[j][1], acc[j][2], acc[j][3], pa0, pa1, pa2, pa3, b0, b1,
                                       acc[j][0] * al0, acc[j][1] * al0, acc[j][2] * al1, acc[j][3] * al1);
                    } else {
                        float d2, d3;
                        mma_bf16_16816(acc[j][0], acc[j][1], d2, d3, pa0, 0u, pa2, 0u, b0, b1, acc[j][0] * al0,
                                       acc[j][1] * al0, 0.f, 0.f);
                    }
                }
            }
        }
    }

    __device__ __forceinline__ void tile(const uint4 (&kf)[2][CH], const uint4 (&vf)[4][CPT / 8], int tb, int n_tok,
                                         float scale_log2, int tq) {
        float s[2][4];
        qk(kf, s);
        uint32_t pa[4];
        float al0, al1;
        softmax(s, tb, n_tok, scale_log2, tq, pa, al0, al1);
        pv(vf, pa, al0, al1);
    }

    // K and V fragments of one tile from a shared-memory stage of K rows then
    // V rows (D channels each); rows past `rows` read the last valid row.  At a
    // row pitch of 2D bytes all rows start in the same bank, so a 16-byte load
    // phase (lanes g even and odd, t = 0..3) would hit few bank groups: lanes of
    // odd g fetch the two 64-byte halves of their K run in swapped order (the
    // phase's two K rows then use both halves of the banks), and lanes of odd t
    // the two 16-byte chunks of their V run; the registers are put back in
    // order after the loads.
    static __device__ __forceinline__ void stage_frags(const uint16_t* ks, const uint16_t* vs, int rows, int gq, int tq,
                                                       uint4 (&kf)[2][CH], uint4 (&vf)[4][CPT / 8]) {
        const bool kx = CH >= 2 && (gq & 1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint16_t* kp = ks + min(8 * h + gq, rows - 1) * D + 8 * tq;
            uint4 t[CH];
#pragma unroll
            for (int s2 = 0; s2 < CH; ++s2) t[s2] = *reinterpret_cast<const uint4*>(kp + 32 * (CH >= 2 ? s2 ^ (int)kx : s2));
#pragma unroll
            for (int s2 = 0; s2 < CH; ++s2) kf[h][s2] = (CH >= 2 && kx) ? t[CH >= 2 ? s2 ^ 1 : s2] : t[s2];
        }
        constexpr int VC = CPT / 8;
        const bool vx = VC >= 2 && (tq & 1);
#pragma unroll
        for (int vi = 0; vi < 4; ++vi) {
            const uint16_t* vp = vs + min(2 * tq + (vi & 1) + 8 * (vi >> 1), rows - 1) * D + CPT * gq;
            uint4 t[VC];
#pragma unroll
            for (int c = 0; c < VC; ++c) t[c] = *reinterpret_cast<const uint4*>(vp + 8 * (VC >= 2 ? c ^ (int)vx : c));
#pragma unroll
            for (int c = 0; c < VC; ++c) vf[vi][c] = (VC >= 2 && vx) ? t[VC >= 2 ? c ^ 1 : c] : t[c];
        }
    }

    // Shared-memory layout of a warp's state: 8*NR rows of D floats.  Lane
    // (g, t) holds channels [2*CPT*t, 2*CPT*(t+1)) of rows g and 8+g (column
    // 2t of n-tile j is channel CPT*2t + j, column 2t+1 is CPT*(2t+1) + j), so
    // it stores them as NC = CPT/2 float4 chunks; its chunk i goes to position
    // NC*t + a rotation of i that differs across the 8 lanes of a 16-byte store
    // phase (t = 0..3, g even and odd), so the phase hits 8 different bank
    // groups rather than one.
    static constexpr int NC = CPT / 2;
    static __device__ __forceinline__ int chunk_pos(int row, int t, int i) {
        if constexpr (D == 128) return 8 * t + ((i + t + 4 * (row & 1)) & 7);
        else return 4 * t + ((i + 2 * (t >> 1) + (row & 1)) & 3);
    }
    // float index of element (row, channel c) in a warp's state area
    static __device__ __forceinline__ int state_idx(int row, int c) {
        const int t = c / (2 * CPT), i = (c % (2 * CPT)) >> 2;
        return row * D + 4 * chunk_pos(row, t, i) + (c & 3);
    }

    // warp state -> shared memory (row sums reduced over the lane quad)
    __device__ __forceinline__ void to_smem(float (*sm_m)[16], float (*sm_l)[16], float* sm_o_w, int warp, int gq,
                                            int tq) {
        static_assert(D == 128 || D == 64, "state layout for d = 64 and 128");
        float a0 = l0, a1 = l1;
        a0 += __shfl_xor_sync(0xffffffffu, a0, 1);
        a0 += __shfl_xor_sync(0xffffffffu, a0, 2);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
        if (tq == 0) {
            sm_m[warp][gq] = m0; sm_l[warp][gq] = a0;
            sm_m[warp][gq + 8] = NR == 2 ? m1 : -INFINITY; sm_l[warp][gq + 8] = NR == 2 ? a1 : 0.f;
        }
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            // chunk i: channels 2*CPT*t + 4i .. +3, from accumulator column 2t (4i < CPT) or 2t+1
            const int j0 = (4 * i) % CPT, e = 4 * i < CPT ? 0 : 1;
            const float4 v = make_float4(acc[j0][e], acc[j0 + 1][e], acc[j0 + 2][e], acc[j0 + 3][e]);
            *reinterpret_cast<float4*>(sm_o_w + gq * D + 4 * chunk_pos(gq, tq, i)) = v;
            if constexpr (NR == 2) {
                const float4 w = make_float4(acc[j0][e + 2], acc[j0 + 1][e + 2], acc[j0 + 2][e + 2], acc[j0 + 3][e + 2]);
                *reinterpret_cast<float4*>(sm_o_w + (gq + 8) * D + 4 * chunk_pos(gq + 8, tq, i)) = w;
            }
        }
    }
};

// Work-item epilogue shared by both kernels: merge the warps' states (already
// in shared memory), write one unnormalised partial for the item, and let the
// CTA that finishes a group's last item (atomic ticket) merge each part and
// fuse the two parts by log-sum-exp.  Called by the nthr compute threads of the
// CTA (threads 0 .. nthr-1), which synchronise on named barrier 1.
template <int D, int NR>
__device__ __forceinline__ void attn_epilogue(float (*sm_m)[16], float (*sm_l)[16], const float* sm_o, int* s_last,
                                              const int4* __restrict__ items, const int32_t* __restrict__ att_first,
                                              const int32_t* __restrict__ att_count, float* __restrict__ part_o,
                                              float* __restrict__ part_ml, uint32_t* __restrict__ done,
                                              float* __restrict__ out_o, float* __restrict__ out_lse,
                                              float* __restrict__ out_o_spec, float* __restrict__ out_lse_spec,
                                              int fuse, int batch, int r, int Hkv, int bg, int nrows,
                                              int64_t item, int nthr) {
    const int tid = threadIdx.x;
    const int b = bg / Hkv, gk = bg % Hkv;
    const int Hq = Hkv * r;
    for (int e = tid; e < nrows * D; e += nthr) {
        const int row = e / D, c = e - row * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w) M = fmaxf(M, sm_m[w][row]);
        float a = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < ATT_WARPS; ++w) {
                const float sc = ex2f(sm_m[w][row] - M);
                a += sc * sm_o[w * 8 * NR * D + WarpAttn<D, NR>::state_idx(row, c)];
                l += sc * sm_l[w][row];
            }
        }
        part_o[(item * nrows + row) * D + c] = a;
        if (c == 0) {
            part_ml[(item * nrows + row) * 2 + 0] = M;
            part_ml[(item * nrows + row) * 2 + 1] = l;
        }
    }
    // the barrier makes the CTA's partial stores visible to thread 0, whose
    // device-scope release fence (cumulative) orders them before its ticket;
    // the last CTA's acquire fence after the ticket orders the merge's loads
    bar_named(1, nthr);
    if (tid == 0) {
        fence_acq_rel_gpu();
        const bool last = atomicAdd(&done[bg], 1u) + 1 == (uint32_t)att_count[bg];
        if (last) fence_acq_rel_gpu();
        *s_last = last;
    }
    bar_named(1, nthr);
    if (!*s_last) return;

    // Merge of the group's partials, per part, by log-sum-exp.  When the group's
    // items fit the table (MI; always, for the work plans built here): the (m, l)
    // of every (item, row) go to shared memory (the warps' state area, free since
    // the partial write), one thread per (part, row) turns them into weights, and
    // every element's partial loads are then independent of one another.  More
    // items: an online merge per element.
    constexpr int MI = D == 128 ? 96 : 48;              // items the table holds
    static_assert(MI * 33 + 64 <= ATT_WARPS * 8 * NR * D, "merge table does not fit the warps' state area");
    float* s_w = const_cast<float*>(sm_o);              // [MI][16] m, then weight, of (item, row)
    float* s_l = s_w + MI * 16;                         // [MI][16] l of (item, row)
    int* s_p = reinterpret_cast<int*>(s_l + MI * 16);   // [MI] part of each item
    float* s_M = reinterpret_cast<float*>(s_p + MI);    // [2][16] maximum of (part, row)
    float* s_L = s_M + 32;                              // [2][16] sum of (part, row)
    const int first = att_first[bg], cnt = att_count[bg];
    const int64_t rows_total = (int64_t)batch * Hq;
    const bool table = cnt <= MI;
    if (table) {
        for (int t = tid; t < cnt * nrows; t += nthr) {
            const int i = t / nrows, row = t - i * nrows;
            const int64_t base = ((int64_t)(first + i) * nrows + row) * 2;
            s_w[i * 16 + row] = __ldcg(part_ml + base);
            s_l[i * 16 + row] = __ldcg(part_ml + base + 1);
            if (row == 0) s_p[i] = __ldg(&items[first + i].y);
        }
        bar_named(1, nthr);
        if (tid < 2 * nrows) {
            const int pp = tid / nrows, row = tid - pp * nrows;
            float Mn = -INFINITY;
            for (int i = 0; i < cnt; ++i)
                if (s_p[i] == pp) Mn = fmaxf(Mn, s_w[i * 16 + row]);
            float L = 0.f;
            for (int i = 0; i < cnt; ++i) {
                if (s_p[i] != pp) continue;
                const float m = s_w[i * 16 + row];
                const float w = m == -INFINITY ? 0.f : ex2f(m - Mn);
                s_w[i * 16 + row] = w;
                L += w * s_l[i * 16 + row];
            }
            s_M[pp * 16 + row] = Mn;
            s_L[pp * 16 + row] = L;
        }
        bar_named(1, nthr);
    }
    for (int e = tid; e < nrows * D; e += nthr) {
        const int row = e / D, c = e - row * D;
        float Mp[2], Lp[2], Ap[2] = {0.f, 0.f};
        if (table) {
            Mp[0] = s_M[row]; Mp[1] = s_M[16 + row];
            Lp[0] = s_L[row]; Lp[1] = s_L[16 + row];
#pragma unroll 4
            for (int i = 0; i < cnt; ++i) {
                const float v = __ldcg(part_o + ((int64_t)(first + i) * nrows + row) * D + c) * s_w[i * 16 + row];
                if (s_p[i]) Ap[1] += v; else Ap[0] += v;
            }
        } else {
            Mp[0] = Mp[1] = -INFINITY;
            Lp[0] = Lp[1] = 0.f;
            for (int i = first; i < first + cnt; ++i) {
                const int64_t base = (int64_t)i * nrows + row;
                const float mi = __ldcg(part_ml + base * 2);
                if (mi == -INFINITY) continue;
                const int pp = __ldg(&items[i].y);
                const float Mn = fmaxf(Mp[pp], mi);
                const float so = ex2f(Mp[pp] - Mn), sn = ex2f(mi - Mn);
                Lp[pp] = Lp[pp] * so + __ldcg(part_ml + base * 2 + 1) * sn;
                Ap[pp] = Ap[pp] * so + __ldcg(part_o + base * D + c) * sn;
                Mp[pp] = Mn;
            }
        }
        const bool spec_row = row >= r;
        const int64_t orow = (int64_t)b * Hq + gk * r + (spec_row ? row - r : row);
        float* dst_o = spec_row ? out_o_spec : out_o;
        float* dst_lse = spec_row ? out_lse_spec : out_lse;
        if (fuse) {
            const float M = fmaxf(Mp[0], Mp[1]);
            float o = 0.f, lse = -INFINITY;
            if (M != -INFINITY) {
                const float w0 = Mp[0] == -INFINITY ? 0.f : ex2f(Mp[0] - M);
                const float w1 = Mp[1] == -INFINITY ? 0.f : ex2f(Mp[1] - M);
                const float L = w0 * Lp[0] + w1 * Lp[1];
                o = (w0 * Ap[0] + w1 * Ap[1]) / L;
                lse = (M + lg2f(L)) * kLn2;
            }
            dst_o[orow * D + c] = o;
            if (c == 0) dst_lse[orow] = lse;
        } else {
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                float o = 0.f, lse = -INFINITY;
                if (Mp[pp] != -INFINITY && Lp[pp] > 0.f) {
                    o = Ap[pp] / Lp[pp];
                    lse = (Mp[pp] + lg2f(Lp[pp])) * kLn2;
                }
                dst_o[(pp * rows_total + orow) * D + c] = o;
                if (c == 0) dst_lse[pp * rows_total + orow] = lse;
            }
        }
    }
    if (tid == 0) done[bg] = 0u;
    // the merge table lives in the warps' state area: no warp may write its
    // next state there before every thread is done reading the table
    bar_named(1, nthr);
}

// ---------------------------------------------------------------------------
// Register-direct kernel: one CTA per work item; each warp loads its tiles'
// K/V fragments straight from global memory with 16-byte loads (next tile
// prefetched into L2).
template <int D, int NR>
__global__ void __launch_bounds__(ATT_WARPS * 32, NR == 1 ? KVO_ATT_MINB_NR1 : 2)
attn_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ q_spec, const uint16_t* __restrict__ bk,
            const uint16_t* __restrict__ bv,
            const uint16_t* __restrict__ wk, const uint16_t* __restrict__ wv, const int32_t* __restrict__ slot,
            const int4* __restrict__ items, const int32_t* __restrict__ att_first, const int32_t* __restrict__ att_count,
            float* __restrict__ part_o, float* __restrict__ part_ml, uint32_t* __restrict__ done,
            float* __restrict__ out_o, float* __restrict__ out_lse, float* __restrict__ out_o_spec,
            float* __restrict__ out_lse_spec, int fuse, int batch, int r, int Hkv, int k,
            int B, int W, int Wcap, const int32_t* __restrict__ w_start, const int32_t* __restrict__ w_len,
            float scale_log2, int32_t* __restrict__ status) {
    using WA = WarpAttn<D, NR>;
    constexpr int CH = WA::CH, CPT = WA::CPT;
    __shared__ float sm_m[ATT_WARPS][16];
    __shared__ float sm_l[ATT_WARPS][16];
    __shared__ __align__(16) float sm_o[ATT_WARPS * 8 * NR * D];
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int4 it = items[blockIdx.x];
    const int bg = it.x, part = it.y, tile0 = it.z, ntiles = it.w;
    const int b = bg / Hkv, gk = bg % Hkv;
    const int Hq = Hkv * r;
    // window: W tokens from slot 0 of [Wcap] rows, or (appendable cache) w_len[bg]
    // tokens of a ring of Wcap rows starting at slot w_start[bg]
    const int ws = w_start ? w_start[bg] : 0;
    const int n_tok = part == 0 ? k * B : (w_len ? w_len[bg] : W);
    // query rows: the r heads of the group, then (co-batched) the r heads of the speculative query
    const int nrows = q_spec ? 2 * r : r;
    auto qrow = [&](int row) -> const uint16_t* {
        return row < r ? q + ((int64_t)b * Hq + gk * r + row) * D : q_spec + ((int64_t)b * Hq + gk * r + row - r) * D;
    };
    WA st;
    {
        const bool v0 = gq < nrows, v1 = NR == 2 && gq + 8 < nrows;
        st.init(v0 ? qrow(gq) : q, v1 ? qrow(gq + 8) : q, v0, v1, tq);
    }
    int bad = 0;
    auto row_ptr = [&](const uint16_t* base_buf, const uint16_t* base_win, int tok) -> const uint16_t* {
        if (part == 0) {
            const int blk = tok / B;
            int s = slot[(int64_t)bg * k + blk];
            if (s < 0 || s >= 2 * k) { bad |= KVO_DEV_BAD_SLOT; s = 0; }
            return base_buf + (((int64_t)bg * 2 * k + s) * B + (tok - blk * B)) * D;
        }
        int slot_w = ws + tok;
        if (slot_w >= Wcap) slot_w -= Wcap;
        return base_win + ((int64_t)bg * Wcap + slot_w) * D;
    };

    for (int tl = warp; tl < ntiles; tl += ATT_WARPS) {
        const int tb = (tile0 + tl) * ATT_TILE;
        if (tb >= n_tok) break;                 // a shorter window than the items cover
        // pull this warp's next tile into L2 while the current one is computed:
        // lane l takes token l & 15, K rows for l < 16 and V rows otherwise (2 lines each)
        if (KVO_ATT_PREFETCH && tl + ATT_WARPS < ntiles) {
            const int ntok = (tile0 + tl + ATT_WARPS) * ATT_TILE + (lane & 15);
            if (ntok < n_tok) {
                const uint16_t* p = row_ptr(lane < 16 ? bk : bv, lane < 16 ? wk : wv, ntok);
#pragma unroll
                for (int off = 0; off < D * 2; off += 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"((const char*)p + off));
            }
        }
        // K rows g and 8+g of the tile
        uint4 kf[2][CH];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int tok = min(tb + 8 * nt + gq, n_tok - 1);
            const uint16_t* kp = row_ptr(bk, wk, tok) + 8 * tq;
#pragma unroll
            for (int s = 0; s < CH; ++s) kf[nt][s] = ldg16(kp + 32 * s);
        }
        // V rows 2t, 2t+1, 2t+8, 2t+9 (channels CPT*g ..)
        uint4 vf[4][CPT / 8];
#pragma unroll
        for (int vi = 0; vi < 4; ++vi) {
            const int tok = min(tb + 2 * tq + (vi & 1) + 8 * (vi >> 1), n_tok - 1);
            const uint16_t* vp = row_ptr(bv, wv, tok) + CPT * gq;
#pragma unroll
            for (int c = 0; c < CPT / 8; ++c) vf[vi][c] = ldg16(vp + 8 * c);
        }
        st.tile(kf, vf, tb, n_tok, scale_log2, tq);
    }
    if (bad && lane == 0) atomicOr(status, bad);
    st.to_smem(sm_m, sm_l, sm_o + warp * 8 * NR * D, warp, gq, tq);
    __syncthreads();
    attn_epilogue<D, NR>(sm_m, sm_l, sm_o, &s_last, items, att_first, att_count, part_o, part_ml, done, out_o,
                         out_lse, out_o_spec, out_lse_spec, fuse, batch, r, Hkv, bg, nrows, blockIdx.x,
                         ATT_WARPS * 32);
}

// ---------------------------------------------------------------------------
// TMA-staged persistent kernel.  The host splits the tiles of all groups
// (sparse part, then window part, group after group) into one contiguous range
// per CTA; the range is cut into work items at part boundaries, so a CTA runs
// one to a few long items and pays the item epilogue (partial write, ticket)
// that rarely.  Within an item warp w takes tiles w, w+4, ..., and every warp
// feeds itself: it keeps its next STG tiles in flight in a private ring of
// shared-memory stages, each filled by cp.async.bulk copies (K rows and V
// rows; one copy per run of contiguous source rows: a run breaks where a
// block's slot does not follow the previous row's, and at the window ring's
// wrap) completing on the stage's mbarrier.  After computing a tile from its
// stage, the warp refills that stage with the tile STG places further down
// its own tile stream, across work items, so copy issue is spread over all
// warps and the loads stay STG tiles ahead of the math.  The fragments are
// read from shared memory with the lane mapping of the register-direct kernel.
// Every mbarrier wait is bounded by the global timer: on expiry the CTA
// records KVO_DEV_TIMEOUT, stops waiting and issues no more copies (its
// results are then invalid; the host sees the status bit), and each warp lets
// the copies it already issued land before it exits.
constexpr int ATT_ITEMS_SMEM = 8;    // work-item headers a CTA keeps in shared memory

template <int D, int NR>
struct AttnTmaCfg {
    // stages per warp: as deep as lets two CTAs share an SM
    static constexpr int STG = D == 128 ? (NR == 1 ? 3 : 2) : 4;
    static constexpr int TILE_BYTES = ATT_TILE * D * 2;                  // one K (or V) tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING = ATT_WARPS * STG * STAGE_BYTES;
    static constexpr int O_FLOATS = ATT_WARPS * 8 * NR * D;
    static constexpr size_t BYTES = (size_t)RING + sizeof(float) * (O_FLOATS + 2 * ATT_WARPS * 16) +
                                    sizeof(uint64_t) * ATT_WARPS * STG + sizeof(int4) * ATT_ITEMS_SMEM + 16;
};

// Bounded wait; false (and the CTA's abort flag set) when the limit passed.
__device__ __forceinline__ bool att_wait(uint32_t mbar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* status, long long limit_ns) {
    if (mbar_try_wait(mbar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (int it = 0;; ++it) {
        if (mbar_try_wait(mbar, parity)) return true;
        if ((it & 63) == 63) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > (uint64_t)limit_ns) {
                *abort_flag = 1;
                atomicOr(status, KVO_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag (a warp's drain before it exits).
__device__ __forceinline__ void att_drain_wait(uint32_t mbar, uint32_t parity, long long limit_ns) {
    if (mbar_try_wait(mbar, parity)) return;
    const uint64_t t0 = global_ns();
    for (int it = 0;; ++it) {
        if (mbar_try_wait(mbar, parity)) return;
        if ((it & 63) == 63 && global_ns() - t0 > (uint64_t)limit_ns) return;
    }
}

// Where one warp stands in its tile stream: work item, tile of the item, and
// the item's fields.  `item == hi` once the stream is exhausted.
struct AttnCursor {
    int item, hi, tl;
    int bg, part, tile0, ntiles, nt, n_tok, ws;
};

// Header of a work item: from the CTA's shared-memory copy of its first
// ATT_ITEMS_SMEM items, else from global memory.
__device__ __forceinline__ int4 item_hdr(const int4* s_items, const int4* __restrict__ items, int lo, int item) {
    return item - lo < ATT_ITEMS_SMEM ? s_items[item - lo] : __ldg(items + item);
}

// Item fields from its header; the window start and length are read only for
// the window part.  `nt` (tiles that hold tokens) is left to cursor_nt, so a
// prefetching caller does not wait for the window length here.
__device__ __forceinline__ void cursor_fields(AttnCursor& c, int4 it, int k, int B, int W,
                                              const int32_t* __restrict__ w_start,
                                              const int32_t* __restrict__ w_len,
                                              const int32_t* __restrict__ sp_cnt) {
    c.bg = it.x; c.part = it.y; c.tile0 = it.z; c.ntiles = it.w;
    c.ws = (c.part == 1 && w_start) ? __ldg(w_start + c.bg) : 0;
    // sparse part: k blocks, or the first sp_cnt[g] entries of the slot list when given
    c.n_tok = c.part == 0 ? (sp_cnt ? min(k, max(0, __ldg(sp_cnt + c.bg))) : k) * B
                          : (w_len ? __ldg(w_len + c.bg) : W);
}
// tiles of the item that hold tokens (a window may be shorter than its items cover)
__device__ __forceinline__ void cursor_nt(AttnCursor& c) {
    c.nt = max(0, min(c.ntiles, (c.n_tok - c.tile0 * ATT_TILE + ATT_TILE - 1) / ATT_TILE));
}

struct ItemSrc {
    const int4* s_items;
    const int4* items;
    int lo, k, B, W;
    const int32_t* w_start;
    const int32_t* w_len;
    const int32_t* sp_cnt;
    __device__ __forceinline__ void load(AttnCursor& c) const {
        cursor_fields(c, item_hdr(s_items, items, lo, c.item), k, B, W, w_start, w_len, sp_cnt);
        cursor_nt(c);
    }
};

// Move to the warp's next tile (tl += ATT_WARPS), into later items when needed.
__device__ __forceinline__ void cursor_next(AttnCursor& c, int warp, const ItemSrc& src) {
    c.tl += ATT_WARPS;
    while (c.tl >= c.nt && c.item < c.hi) {
        if (++c.item == c.hi) break;
        src.load(c);
        c.tl = warp;
    }
}

__device__ __forceinline__ void cursor_first(AttnCursor& c, int lo, int hi, int warp, const ItemSrc& src) {
    c.item = lo; c.hi = hi; c.tl = warp; c.nt = 0;
    if (c.item >= c.hi) return;
    src.load(c);
    while (c.tl >= c.nt) {
        if (++c.item == c.hi) break;
        src.load(c);
    }
}

// Slot of the gathered block holding this lane's row (lane & 15) of the
// cursor's tile (0 where the row does not exist or lies in the window).
__device__ __forceinline__ int cursor_slot(const AttnCursor& c, const int32_t* __restrict__ slot, int k, int B,
                                           int row) {
    if (c.item >= c.hi || c.part != 0) return 0;
    const int tok = (c.tile0 + c.tl) * ATT_TILE + row;
    if (tok >= c.n_tok) return 0;
    return __ldg(slot + (int64_t)c.bg * k + tok / B);
}

// Copy the cursor's tile into a stage: lane j copies row j & 15 of the K tile
// (j < 16) or of the V tile (j >= 16); `sl` is the lane's cursor_slot.  With
// `skip` the stage is announced but nothing is copied, so its barrier never
// completes (the bounded-wait test).
template <int D>
__device__ __forceinline__ void tile_copy(const AttnCursor& c, int sl, unsigned char* stage, uint32_t fb,
                                          const uint16_t* __restrict__ bk, const uint16_t* __restrict__ bv,
                                          const uint16_t* __restrict__ wk, const uint16_t* __restrict__ wv, int k,
                                          int B, int Wcap, int& bad, bool skip) {
    const int lane = threadIdx.x & 31, kv = lane >> 4, row = lane & 15;
    const int tb = (c.tile0 + c.tl) * ATT_TILE;
    const int rows = min(ATT_TILE, c.n_tok - tb);
    if (lane == 0) mbar_expect_tx(fb, (uint32_t)(rows * D * 2 * 2));
    __syncwarp();
    const int tok = tb + row;
    const bool valid = row < rows;
    const uint16_t* src;
    bool start;
    if (c.part == 0) {
        const int blk = tok / B, off = tok - blk * B;
        if (valid && (sl < 0 || sl >= 2 * k)) { bad |= KVO_DEV_BAD_SLOT; sl = 0; }
        const int sl_prev = __shfl_up_sync(0xffffffffu, sl, 1);
        src = (kv ? bv : bk) + (((int64_t)c.bg * 2 * k + sl) * B + off) * D;
        start = valid && (row == 0 || (off == 0 && sl != sl_prev + 1));
    } else {
        int sw = c.ws + tok;
        if (sw >= Wcap) sw -= Wcap;
        src = (kv ? wv : wk) + ((int64_t)c.bg * Wcap + sw) * D;
        start = valid && (row == 0 || sw == 0);
    }
    const unsigned starts = (__ballot_sync(0xffffffffu, start) >> (kv * 16)) & 0xffffu;
    if (start && !skip) {
        const unsigned later = starts & ~((2u << row) - 1u);
        const int next = later ? __ffs(later) - 1 : rows;
        bulk_load(smem_u32(stage + kv * (ATT_TILE * D * 2) + row * D * 2), src, (uint32_t)((next - row) * D * 2),
                  fb);
    }
}

template <int D, int NR>
__global__ void __launch_bounds__(ATT_WARPS * 32, 2)
attn_tma_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ q_spec,
                const uint16_t* __restrict__ bk, const uint16_t* __restrict__ bv, const uint16_t* __restrict__ wk,
                const uint16_t* __restrict__ wv, const int32_t* __restrict__ slot, const int4* __restrict__ items,
                const int32_t* __restrict__ cta_first, const int32_t* __restrict__ att_first,
                const int32_t* __restrict__ att_count, float* __restrict__ part_o, float* __restrict__ part_ml,
                uint32_t* __restrict__ done, float* __restrict__ out_o, float* __restrict__ out_lse,
                float* __restrict__ out_o_spec, float* __restrict__ out_lse_spec, int fuse, int batch, int r,
                int Hkv, int k, int B, int W, int Wcap, const int32_t* __restrict__ w_start,
                const int32_t* __restrict__ w_len, const int32_t* __restrict__ sp_cnt, int dep_wait,
                float scale_log2, int32_t* __restrict__ status, long long wait_ns, int skip_tile) {
    using WA = WarpAttn<D, NR>;
    using CF = AttnTmaCfg<D, NR>;
    constexpr int CH = WA::CH, CPT = WA::CPT, STG = CF::STG;
    constexpr int NTHR = ATT_WARPS * 32;
    extern __shared__ __align__(128) unsigned char smem[];
    float* sm_o = reinterpret_cast<float*>(smem + CF::RING);
    float (*sm_m)[16] = reinterpret_cast<float (*)[16]>(sm_o + CF::O_FLOATS);
    float (*sm_l)[16] = sm_m + ATT_WARPS;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm_l + ATT_WARPS);   // [ATT_WARPS][STG]
    int4* s_items = reinterpret_cast<int4*>(full + ATT_WARPS * STG);  // [ATT_ITEMS_SMEM]
    int* s_last = reinterpret_cast<int*>(s_items + ATT_ITEMS_SMEM);
    volatile int* s_abort = s_last + 1;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3, row = lane & 15;
    const int lo = cta_first[blockIdx.x], hi = cta_first[blockIdx.x + 1];
    if (tid < ATT_WARPS * STG) mbar_init(smem_u32(&full[tid]), 1);
    if (tid < ATT_ITEMS_SMEM && lo + tid < hi) s_items[tid] = items[lo + tid];
    if (tid == 0) *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    const int Hq = Hkv * r;
    const int nrows = q_spec ? 2 * r : r;
    const ItemSrc src{s_items, items, lo, k, B, W, w_start, w_len, sp_cnt};
    unsigned char* ring = smem + warp * STG * CF::STAGE_BYTES;
    uint64_t* wfull = full + warp * STG;
    int bad = 0;

    // issue cursor: STG tiles ahead of the math in this warp's tile stream
    AttnCursor ic;
    cursor_first(ic, lo, hi, warp, src);
    int isl = cursor_slot(ic, slot, k, B, row);
    int64_t nissue = 0, ncons = 0;
    auto issue = [&]() {
        // nothing more is issued once the CTA gave up (lane 0's view, so the whole warp agrees)
        if (ic.item >= ic.hi || __shfl_sync(0xffffffffu, *s_abort, 0)) return;
        const int st = (int)(nissue % STG);
        tile_copy<D>(ic, isl, ring + st * CF::STAGE_BYTES, smem_u32(&wfull[st]), bk, bv, wk, wv, k, B, Wcap, bad,
                     blockIdx.x == 0 && warp == 0 && nissue == skip_tile);
        ++nissue;
        cursor_next(ic, warp, src);
        isl = cursor_slot(ic, slot, k, B, row);
    };
    // prologue: the cursors of the warp's first STG tiles, then their slot
    // loads side by side, then the copies -- rather than STG issues that each
    // wait for the slot load the previous one started (the launch ramp)
    {
        AttnCursor pc[STG];
        int ps[STG];
        pc[0] = ic;
#pragma unroll
        for (int i = 1; i < STG; ++i) {
            pc[i] = pc[i - 1];
            cursor_next(pc[i], warp, src);
        }
#pragma unroll
        for (int i = 0; i < STG; ++i) ps[i] = cursor_slot(pc[i], slot, k, B, row);
#pragma unroll
        for (int i = 0; i < STG; ++i) {
            if (pc[i].item >= pc[i].hi || __shfl_sync(0xffffffffu, *s_abort, 0)) break;
            tile_copy<D>(pc[i], ps[i], ring + i * CF::STAGE_BYTES, smem_u32(&wfull[i]), bk, bv, wk, wv, k, B, Wcap,
                         bad, blockIdx.x == 0 && warp == 0 && nissue == skip_tile);
            ++nissue;
        }
        ic = pc[STG - 1];
        cursor_next(ic, warp, src);
        isl = cursor_slot(ic, slot, k, B, row);
    }

    // the next item's fields and Q words, fetched one item ahead
    const bool v0 = gq < nrows, v1 = NR == 2 && gq + 8 < nrows;
    AttnCursor nc;
    uint4 nq0[CH], nq1[CH];
    auto fetch = [&](int item) {
        nc.item = item; nc.hi = hi; nc.tl = warp;
        cursor_fields(nc, item_hdr(s_items, items, lo, item), k, B, W, w_start, w_len, sp_cnt);
        const int b = nc.bg / Hkv, gk = nc.bg % Hkv;
        auto qrow = [&](int rr) -> const uint16_t* {
            return rr < r ? q + ((int64_t)b * Hq + gk * r + rr) * D : q_spec + ((int64_t)b * Hq + gk * r + rr - r) * D;
        };
        WA::load_q(v0 ? qrow(gq) : q, v1 ? qrow(gq + 8) : q, v0, v1, tq, nq0, nq1);
    };
    if (lo < hi) fetch(lo);

    for (int item = lo; item < hi; ++item) {
        AttnCursor cc = nc;                  // this item, from this warp's view
        cursor_nt(cc);
        WA stt;
        stt.init_from(nq0, nq1);
        if (item + 1 < hi) fetch(item + 1);
        for (int tl = warp; tl < cc.nt; tl += ATT_WARPS) {
            const int st = (int)(ncons % STG);
            if (!*s_abort) att_wait(smem_u32(&wfull[st]), (uint32_t)((ncons / STG) & 1), s_abort, status, wait_ns);
            ++ncons;
            const int tb = (cc.tile0 + tl) * ATT_TILE;
            const int rows = min(ATT_TILE, cc.n_tok - tb);
            const uint16_t* ks = reinterpret_cast<const uint16_t*>(ring + st * CF::STAGE_BYTES);
            // rows past the tile's end hold stale data: the last valid row is read instead
            uint4 kf[2][CH];
            uint4 vf[4][CPT / 8];
            WA::stage_frags(ks, ks + ATT_TILE * D, rows, gq, tq, kf, vf);
            stt.tile(kf, vf, tb, cc.n_tok, scale_log2, tq);
            // the stage's shared-memory reads are done (their values fed the mma):
            // order them before the async-proxy refill of the same stage
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue();
        }
        stt.to_smem(sm_m, sm_l, sm_o + warp * 8 * NR * D, warp, gq, tq);
        bar_named(1, NTHR);
        attn_epilogue<D, NR>(sm_m, sm_l, sm_o, s_last, items, att_first, att_count, part_o, part_ml, done, out_o,
                             out_lse, out_o_spec, out_lse_spec, fuse, batch, r, Hkv, cc.bg, nrows, item, NTHR);
    }
    if (bad) atomicOr(status, bad);
    // Before the warp exits, every copy it issued has landed: without an abort
    // it waited for each; after one it may have stopped waiting, so it checks
    // -- with bounded waits -- its last STG copies, the only ones that can
    // still be in flight, and no bulk copy is left writing into the shared
    // memory of a CTA that has finished.
    if (lane == 0)
        for (int64_t s2 = nissue > STG ? nissue - STG : 0; s2 < nissue; ++s2)
            att_drain_wait(smem_u32(&wfull[s2 % STG]), (uint32_t)((s2 / STG) & 1), wait_ns);
    __syncwarp();
    // launched as a programmatic dependent: this grid completes only after the
    // grid it depends on, so the launches behind it see that grid's writes
    if (dep_wait && tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Group-split cluster kernel (fused output only).  Each (request, KV head)
// group gets a cluster of S CTAs that split the group's tiles (sparse part,
// then window part): warp j of the cluster (j = rank * 4 + warp) takes the
// blocks of STG consecutive tiles j, j + 4S, j + 8S, ... .  A warp copies its
// tiles into its ring of STG shared-memory stages with bulk copies (as in the
// persistent kernel) and refills a stage right after computing it.  The
// fused output is the softmax over the union of the two parts (log-sum-exp
// merge of the parts is that softmax, regrouped), so a warp keeps one
// online-softmax state whatever part its tiles come from, and no CTA has a
// per-item epilogue: after its last tile the warps' states are merged in the
// CTA's own shared memory, the cluster synchronises once, and each CTA merges
// a 1/S slice of the group's output elements by reading the S CTA states
// through distributed shared memory -- no partials in global memory, no
// ticket, no device-scope fence.  A second cluster barrier keeps every CTA's
// shared memory alive until the last remote read.  The group's slot list is
// staged in shared memory by asynchronous copies that overlap the first tile
// copies (whose slots are read from global memory).  Two stages per warp and
// two CTAs per SM measured faster than deeper rings or three CTAs per SM, and
// a tile counter drawn through a shared-memory atomic (to balance a cluster's
// CTAs dynamically) cost more than the imbalance it removed.  Waits are
// bounded as in the persistent kernel; a CTA that gave up still reaches both
// cluster barriers.
template <int D, int NR>
struct AttnCluCfg {
    static constexpr int STG = D == 128 ? 2 : 4;                          // stages per warp
    static constexpr int STAGE_BYTES = 2 * ATT_TILE * D * 2;              // K and V tile
    static constexpr int RING = ATT_WARPS * STG * STAGE_BYTES;
    static constexpr int O_FLOATS = ATT_WARPS * 8 * NR * D;               // warp states, in the idle ring
    static constexpr int SLOT_CAP = 4096;                                 // slot entries staged in shared memory
    static_assert(sizeof(float) * (O_FLOATS + 32 + 16 * D + 16 * 8) <= (size_t)RING,
                  "end-phase state does not fit the ring");
    // ring | m, l [ATT_WARPS][16] each | full [ATT_WARPS][STG] | tile of each stage [ATT_WARPS][STG] |
    // abort flag (16 B) | slot table [SLOT_CAP]: 82 KB, two CTAs per SM
    static constexpr size_t BYTES = (size_t)RING + sizeof(float) * 2 * ATT_WARPS * 16 +
                                    sizeof(uint64_t) * ATT_WARPS * STG + sizeof(int) * ATT_WARPS * STG + 16 +
                                    sizeof(int) * SLOT_CAP;
};
constexpr int ATT_CLU_MAX = 8;       // CTAs per group (portable cluster size)

template <int D, int NR>
__global__ void __launch_bounds__(ATT_WARPS * 32, 2)
attn_cluster_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ q_spec,
                    const uint16_t* __restrict__ bk, const uint16_t* __restrict__ bv,
                    const uint16_t* __restrict__ wk, const uint16_t* __restrict__ wv,
                    const int32_t* __restrict__ slot, float* __restrict__ out_o, float* __restrict__ out_lse,
                    float* __restrict__ out_o_spec, float* __restrict__ out_lse_spec, int r, int Hkv, int k, int B,
                    int W, int Wcap, const int32_t* __restrict__ w_start, const int32_t* __restrict__ w_len,
                    const int32_t* __restrict__ sp_cnt, int dep_mode, float scale_log2,
                    int32_t* __restrict__ status, long long wait_ns, int skip_tile) {
    using WA = WarpAttn<D, NR>;
    using CF = AttnCluCfg<D, NR>;
    constexpr int CH = WA::CH, CPT = WA::CPT, STG = CF::STG;
    constexpr int NTHR = ATT_WARPS * 32;
    extern __shared__ __align__(128) unsigned char smem[];
    float (*sm_m)[16] = reinterpret_cast<float (*)[16]>(smem + CF::RING);
    float (*sm_l)[16] = sm_m + ATT_WARPS;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm_l + ATT_WARPS);     // [ATT_WARPS][STG]
    int* s_tile = reinterpret_cast<int*>(full + ATT_WARPS * STG);       // [ATT_WARPS][STG] tile in each stage
    volatile int* s_abort = s_tile + ATT_WARPS * STG;
    int* s_slot = s_tile + ATT_WARPS * STG + 4;                         // [SLOT_CAP]
    float* sm_o = reinterpret_cast<float*>(smem);                      // end phase only (ring idle)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3, row = lane & 15;
    const uint32_t S = max(1u, cluster_size()), rank = S > 1 ? cluster_rank() : 0u;
    const int bg = (int)(blockIdx.x / S);
    const bool tab = k <= CF::SLOT_CAP;
    if (tid < ATT_WARPS * STG) mbar_init(smem_u32(&full[tid]), 1);
    if (tid == 0) *s_abort = 0;
    // dep_mode 2: launched as a programmatic dependent of the kernel before it
    // on the stream, which may have written any input -- nothing is read before
    // it is done (0: an ordinary launch)
    if (dep_mode == 2) asm volatile("griddepcontrol.wait;" ::: "memory");
    // the group's slot list into shared memory, asynchronously (read after the first copies are out)
    if (tab) {
        const int32_t* src = slot + (int64_t)bg * k;
        for (int i = tid; i < k; i += NTHR)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s_slot + i)), "l"(src + i) : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    // the group's tiles: sparse part (tiles [0, t_sp)), then window part
    const int n_sp = (sp_cnt ? min(k, max(0, __ldg(sp_cnt + bg))) : k) * B;
    const int n_w = max(0, w_len ? __ldg(w_len + bg) : W);
    const int ws = w_start ? __ldg(w_start + bg) : 0;
    const int t_sp = (n_sp + ATT_TILE - 1) / ATT_TILE;
    const int T = t_sp + (n_w + ATT_TILE - 1) / ATT_TILE;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    const int Hq = Hkv * r;
    const int nrows = q_spec ? 2 * r : r;
    unsigned char* ring = smem + warp * STG * CF::STAGE_BYTES;
    uint64_t* wfull = full + warp * STG;
    int* wtile = s_tile + warp * STG;
    int bad = 0;
    const bool skip_cta = blockIdx.x == 0 && warp == 0;

    // tile t as the cursor the copy routine takes
    auto cur = [&](int t) {
        AttnCursor c;
        c.item = 0; c.hi = 1; c.tl = 0; c.bg = bg; c.ntiles = 1; c.nt = 1;
        c.part = t < t_sp ? 0 : 1;
        c.tile0 = c.part ? t - t_sp : t;
        c.n_tok = c.part ? n_w : n_sp;
        c.ws = c.part ? ws : 0;
        return c;
    };
    // slot of this lane's row of tile t (0 outside the sparse part)
    auto slot_of = [&](int t, bool from_tab) -> int {
        if (t >= t_sp) return 0;
        const int tok = t * ATT_TILE + row;
        if (tok >= n_sp) return 0;
        return from_tab ? s_slot[tok / B] : __ldg(slot + (int64_t)bg * k + tok / B);
    };
    int64_t nissue = 0, ncons = 0;
    auto copy = [&](int t, int sl) {
        const int st = (int)(nissue % STG);
        if (lane == 0) wtile[st] = t;
        tile_copy<D>(cur(t), sl, ring + st * CF::STAGE_BYTES, smem_u32(&wfull[st]), bk, bv, wk, wv, k, B, Wcap, bad,
                     skip_cta && nissue == skip_tile);
        ++nissue;
    };
    // this warp's tiles: blocks of STG consecutive tiles (one gathered block
    // when B = 32), block j of the cluster's warp j, j + 4S, j + 8S, ...
    const int stride = (int)S * ATT_WARPS * STG;
    int next = ((int)rank * ATT_WARPS + warp) * STG;
    // the first block: slots straight from global memory, copies out
    {
        int ps[STG];
#pragma unroll
        for (int i = 0; i < STG; ++i) ps[i] = next + i < T ? slot_of(next + i, false) : 0;
#pragma unroll
        for (int i = 0; i < STG; ++i)
            if (next + i < T) copy(next + i, ps[i]);
        next += stride;
    }
    if (tab) asm volatile("cp.async.wait_all;" ::: "memory");
    bar_named(1, NTHR);                      // slot table visible to every warp
    int nidx = 0;
    auto refill = [&]() {
        if (__shfl_sync(0xffffffffu, *s_abort, 0)) return;      // lane 0's view: the warp agrees
        const int t = next + nidx;
        if (t >= T) return;
        if (++nidx == STG) { nidx = 0; next += stride; }
        copy(t, slot_of(t, tab));
    };

    // one state over all the group's rows, whatever part each tile comes from
    WA stt;
    {
        const int b = bg / Hkv, gk = bg % Hkv;
        auto qrow = [&](int rr) -> const uint16_t* {
            return rr < r ? q + ((int64_t)b * Hq + gk * r + rr) * D : q_spec + ((int64_t)b * Hq + gk * r + rr - r) * D;
        };
        const bool v0 = gq < nrows, v1 = NR == 2 && gq + 8 < nrows;
        stt.init(v0 ? qrow(gq) : q, v1 ? qrow(gq + 8) : q, v0, v1, tq);
    }
    while (ncons < nissue) {
        const int st = (int)(ncons % STG);
        if (!*s_abort) att_wait(smem_u32(&wfull[st]), (uint32_t)((ncons / STG) & 1), s_abort, status, wait_ns);
        ++ncons;
        const int t = wtile[st];
        const bool sp = t < t_sp;
        const int tb = (sp ? t : t - t_sp) * ATT_TILE, n_tok = sp ? n_sp : n_w;
        const int rows = min(ATT_TILE, n_tok - tb);
        const uint16_t* ks = reinterpret_cast<const uint16_t*>(ring + st * CF::STAGE_BYTES);
        uint4 kf[2][CH];
        uint4 vf[4][CPT / 8];
        WA::stage_frags(ks, ks + ATT_TILE * D, rows, gq, tq, kf, vf);
        stt.tile(kf, vf, tb, n_tok, scale_log2, tq);
        // the stage's reads are done: order them before the async-proxy refill
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        refill();
    }
    // the kernel behind this one on the stream may be scheduled now (it waits
    // for this grid to finish before it reads anything)
    if (dep_mode == 2) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (bad) atomicOr(status, bad);
    // every copy has landed before the ring is reused (bounded, as in the persistent kernel)
    if (lane == 0)
        for (int64_t s2 = nissue > STG ? nissue - STG : 0; s2 < nissue; ++s2)
            att_drain_wait(smem_u32(&wfull[s2 % STG]), (uint32_t)((s2 / STG) & 1), wait_ns);
    __syncthreads();
    stt.to_smem(sm_m, sm_l, sm_o + warp * 8 * NR * D, warp, gq, tq);
    __syncthreads();

    // this CTA's state, its warps merged: max and mass per row (log2 domain)
    // and the unnormalised sum per element, in the ring after the warp states
    float* c_m = sm_o + CF::O_FLOATS;
    float* c_l = c_m + 16;
    float* c_a = c_l + 16;
    for (int e = tid; e < nrows * D; e += NTHR) {
        const int rr = e / D, c = e - rr * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w) M = fmaxf(M, sm_m[w][rr]);
        float a = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < ATT_WARPS; ++w) {
                const float sc = ex2f(sm_m[w][rr] - M);
                a += sc * sm_o[w * 8 * NR * D + WA::state_idx(rr, c)];
                l += sc * sm_l[w][rr];
            }
        }
        c_a[rr * D + c] = a;
        if (c == 0) { c_m[rr] = M; c_l[rr] = l; }
    }
    if (S > 1) cluster_barrier(); else __syncthreads();

    // per row: the weight of each CTA state (its share of the row's softmax
    // mass, normalised) and the row's log-sum-exp, written by the first CTA
    const int b = bg / Hkv, gk = bg % Hkv;
    float* s_wt = c_a + 16 * D;              // [16][ATT_CLU_MAX]
    if (tid < nrows) {
        float ms[ATT_CLU_MAX], ls[ATT_CLU_MAX];
#pragma unroll
        for (int s2 = 0; s2 < ATT_CLU_MAX; ++s2)
            if (s2 < (int)S) {
                ms[s2] = S > 1 ? ld_cluster_f32(c_m + tid, s2) : c_m[tid];
                ls[s2] = S > 1 ? ld_cluster_f32(c_l + tid, s2) : c_l[tid];
            }
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < ATT_CLU_MAX; ++s2)
            if (s2 < (int)S) M = fmaxf(M, ms[s2]);
        float L = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < ATT_CLU_MAX; ++s2)
            if (s2 < (int)S) {
                ms[s2] = (M == -INFINITY || ms[s2] == -INFINITY) ? 0.f : ex2f(ms[s2] - M);
                L += ms[s2] * ls[s2];
            }
        const float inv = M == -INFINITY ? 0.f : __frcp_rn(L);
#pragma unroll
        for (int s2 = 0; s2 < ATT_CLU_MAX; ++s2)
            if (s2 < (int)S) s_wt[tid * ATT_CLU_MAX + s2] = ms[s2] * inv;
        if (rank == 0) {
            const bool spec_row = tid >= r;
            const int64_t orow = (int64_t)b * Hq + gk * r + (spec_row ? tid - r : tid);
            (spec_row ? out_lse_spec : out_lse)[orow] = M == -INFINITY ? -INFINITY : (M + lg2f(L)) * kLn2;
        }
    }
    __syncthreads();
    // the group's output: CTA `rank` merges elements rank*NTHR + tid, + S*NTHR, ...
    // (each element's S remote loads issued together)
    for (int e = (int)rank * NTHR + tid; e < nrows * D; e += (int)S * NTHR) {
        const int rr = e / D, c = e - rr * D;
        float as[ATT_CLU_MAX];
#pragma unroll
        for (int s2 = 0; s2 < ATT_CLU_MAX; ++s2)
            if (s2 < (int)S) as[s2] = S > 1 ? ld_cluster_f32(c_a + rr * D + c, s2) : c_a[rr * D + c];
        float o = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < ATT_CLU_MAX; ++s2)
            if (s2 < (int)S) o += s_wt[rr * ATT_CLU_MAX + s2] * as[s2];
        const bool spec_row = rr >= r;
        const int64_t orow = (int64_t)b * Hq + gk * r + (spec_row ? rr - r : rr);
        (spec_row ? out_o_spec : out_o)[orow * D + c] = o;
    }
    // no CTA leaves (and frees its shared memory) while another may still read it
    if (S > 1) cluster_barrier();
}

template <int D, int NR>
static cudaError_t tma_attr(int* per_sm, int* clu_per_sm) {
    cudaError_t e = cudaFuncSetAttribute(attn_tma_kernel<D, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)AttnTmaCfg<D, NR>::BYTES);
    if (e != cudaSuccess) return e;
    using CC = AttnCluCfg<D, NR>;
    e = cudaFuncSetAttribute(attn_cluster_kernel<D, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CC::BYTES);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(clu_per_sm, attn_cluster_kernel<D, NR>, ATT_WARPS * 32,
                                                      CC::BYTES);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, attn_tma_kernel<D, NR>, ATT_WARPS * 32,
                                                         AttnTmaCfg<D, NR>::BYTES);
}

// Shared-memory attribute of the TMA-staged kernel; SMs of the device and
// CTAs of the kernel per SM (the smaller count of its two query-row variants).
cudaError_t prepare_attention(Ctx& c) {
    int dev = 0, sms = 0, p1 = 0, p2 = 0, q1 = 0, q2 = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (c.d == 128) {
        if ((e = tma_attr<128, 1>(&p1, &q1)) != cudaSuccess || (e = tma_attr<128, 2>(&p2, &q2)) != cudaSuccess)
            return e;
    } else {
        if ((e = tma_attr<64, 1>(&p1, &q1)) != cudaSuccess || (e = tma_attr<64, 2>(&p2, &q2)) != cudaSuccess)
            return e;
    }
    c.tma_per_sm = std::max(1, std::min(p1, p2));
    c.clu_per_sm = std::max(1, std::min(q1, q2));
    c.n_sms = std::max(1, sms);
    return cudaSuccess;
}

template <int D, int NR>
static cudaError_t launch_tma(const Ctx& c, const Ctx::TmaPlan& pl, int buf, const void* q, const void* q_spec,
                              const uint16_t* wk, const uint16_t* wv, const int32_t* slot, float* o, float* lse,
                              float* o_spec, float* lse_spec, int fuse, cudaStream_t s, const int32_t* sp_cnt,
                              bool pdl, float scale_log2, float* part_o, float* part_ml, uint32_t* done) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(ATT_WARPS * 32);
    cfg.dynamicSmemBytes = AttnTmaCfg<D, NR>::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_tma_kernel<D, NR>, (const uint16_t*)q, (const uint16_t*)q_spec,
                              (const uint16_t*)c.buf_k(buf), (const uint16_t*)c.buf_v(buf), wk, wv, slot,
                              (const int4*)pl.items, (const int32_t*)pl.cta, (const int32_t*)pl.first,
                              (const int32_t*)pl.count, part_o, part_ml, done, o, lse, o_spec,
                              lse_spec, fuse, c.batch, c.r, c.Hkv, c.k, c.B, c.W, c.Wcap, (const int32_t*)c.g_wstart,
                              (const int32_t*)c.g_wlen, sp_cnt, pdl ? 1 : 0, scale_log2, c.status,
                              (long long)c.att_wait_ns, c.att_skip_tile);
}

template <int D, int NR>
static cudaError_t launch_cluster(const Ctx& c, int S, int buf, const void* q, const void* q_spec,
                                  const uint16_t* wk, const uint16_t* wv, const int32_t* slot, float* o, float* lse,
                                  float* o_spec, float* lse_spec, cudaStream_t s, const int32_t* sp_cnt,
                                  int dep_mode, float scale_log2) {
    const bool pdl = dep_mode == 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(c.G * S));
    cfg.blockDim = dim3(ATT_WARPS * 32);
    cfg.dynamicSmemBytes = AttnCluCfg<D, NR>::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<D, NR>, (const uint16_t*)q, (const uint16_t*)q_spec,
                              (const uint16_t*)c.buf_k(buf), (const uint16_t*)c.buf_v(buf), wk, wv, slot, o, lse,
                              o_spec, lse_spec, c.r, c.Hkv, c.k, c.B, c.W, c.Wcap, (const int32_t*)c.g_wstart,
                              (const int32_t*)c.g_wlen, sp_cnt, dep_mode, scale_log2, c.status,
                              (long long)c.att_wait_ns, c.att_skip_tile);
}

cudaError_t launch_attention(const Ctx& c, int layer, int buf, const void* q, const void* q_spec, const int32_t* slot,
                             float* o, float* lse, float* o_spec, float* lse_spec, int fuse, cudaStream_t s,
                             bool in_step, const int32_t* sp_cnt, bool pdl, int scratch) {
    // the scratch set of the work-item kernels: partial results and tickets
    const size_t prow = 2 * c.r <= 16 ? 2 * c.r : c.r;
    float* part_o = c.att_part_o + (scratch ? (size_t)c.att_part_cap * prow * c.d : 0);
    float* part_ml = c.att_part_ml + (scratch ? (size_t)c.att_part_cap * prow * 2 : 0);
    uint32_t* done = c.att_done + (scratch ? c.G : 0);
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.d));
    const uint16_t* wk = c.W > 0 ? c.k_win[layer] : nullptr;
    const uint16_t* wv = c.W > 0 ? c.v_win[layer] : nullptr;
    const int nrows = q_spec ? 2 * c.r : c.r;
    const Ctx::TmaPlan& pl = c.tma[in_step ? 1 : 0];
    // A dependent launch that waits for its predecessor at its end (pdl) keeps
    // its CTAs resident until then, so it must fit in one wave: the persistent
    // kernel's plan is exactly the resident slots, a cluster grid may not be.
    if (c.att_impl == 2 && fuse && c.clu_use[in_step ? 1 : 0] && !pdl) {
        const int S = c.clu_S[in_step ? 1 : 0];
        // a standalone call: a dependent of whatever ran before it on the stream
        // (inside a decode step an early launch could hold SMs the step's gathers
        // are about to take)
        const int dep_mode = c.att_pdl && !in_step ? 2 : 0;
#define KVO_CLU(D_, NR_) \
        launch_cluster<D_, NR_>(c, S, buf, q, q_spec, wk, wv, slot, o, lse, o_spec, lse_spec, s, sp_cnt, dep_mode, \
                                scale_log2)
        if (c.d == 128) return nrows <= 8 ? KVO_CLU(128, 1) : KVO_CLU(128, 2);
        return nrows <= 8 ? KVO_CLU(64, 1) : KVO_CLU(64, 2);
#undef KVO_CLU
    }
    // impl 2 with separate parts (fuse 0), with too few groups to fill the
    // device, or launched to wait at its end, uses the persistent kernel
    if (c.att_impl >= 1) {
#define KVO_TMA(D_, NR_) \
        launch_tma<D_, NR_>(c, pl, buf, q, q_spec, wk, wv, slot, o, lse, o_spec, lse_spec, fuse, s, sp_cnt, pdl, \
                            scale_log2, part_o, part_ml, done)
        if (c.d == 128) return nrows <= 8 ? KVO_TMA(128, 1) : KVO_TMA(128, 2);
        return nrows <= 8 ? KVO_TMA(64, 1) : KVO_TMA(64, 2);
#undef KVO_TMA
    }
    // partial slot lists and dependent launches exist in the TMA-staged kernel only
    if (sp_cnt || pdl) return cudaErrorInvalidValue;
#define KVO_ATT(D_, NR_)                                                                                         \
    attn_kernel<D_, NR_><<<c.n_att_items, ATT_WARPS * 32, 0, s>>>(                                               \
        (const uint16_t*)q, (const uint16_t*)q_spec, c.buf_k(buf), c.buf_v(buf), wk, wv, slot, c.att_items,       \
        c.att_first, c.att_count, part_o, part_ml, done, o, lse, o_spec, lse_spec, fuse,                          \
        c.batch, c.r, c.Hkv, c.k, c.B, c.W, c.Wcap, c.g_wstart, c.g_wlen, scale_log2, c.status)
    if (c.d == 128) {
        if (nrows <= 8) KVO_ATT(128, 1); else KVO_ATT(128, 2);
    } else {
        if (nrows <= 8) KVO_ATT(64, 1); else KVO_ATT(64, 2);
    }
#undef KVO_ATT
    return cudaGetLastError();
}

// --------------------------------------------------- attention over a few more blocks
// Attention of each group's r query rows over the first cnt[g] entries of a
// slot list, merged by log-sum-exp with a prior part (prior_o, prior_lse: the
// attention over the group's other keys) into out_o / out_lse.  A decode step
// whose blocks were resident but for a few fetched ones attends to the
// resident ones beside the fetch and to the fetched ones here, after it.
// Grid (G, S): the S CTAs of a group take its tiles round-robin (CTA s, warp
// w: tiles 4s + w, 4s + w + 4S, ...; register-direct, each warp's next tile
// pulled into L2 while it computes the current one), so a group with many
// fetched blocks still spreads over 4S warps.  With S > 1 each CTA leaves an
// unnormalised partial and the last one to finish (atomic ticket) merges them.
template <int D, int NR>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attn_merge_part_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ bk,
                       const uint16_t* __restrict__ bv, const int32_t* __restrict__ slot,
                       const int32_t* __restrict__ cnt, const float* __restrict__ prior_o,
                       const float* __restrict__ prior_lse, float* __restrict__ out_o, float* __restrict__ out_lse,
                       float* __restrict__ part_o, float* __restrict__ part_ml, uint32_t* __restrict__ done, int r,
                       int Hkv, int k, int B, float scale_log2, int32_t* __restrict__ status) {
    using WA = WarpAttn<D, NR>;
    constexpr int CH = WA::CH, CPT = WA::CPT;
    __shared__ float sm_m[ATT_WARPS][16];
    __shared__ float sm_l[ATT_WARPS][16];
    __shared__ __align__(16) float sm_o[ATT_WARPS * 8 * NR * D];
    __shared__ int s_last;
    const int bg = blockIdx.x, S = gridDim.y, sl_i = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int b = bg / Hkv, gk = bg % Hkv, Hq = Hkv * r;
    int bad = 0;
    int n = cnt[bg];
    if (n < 0 || n > k) { bad |= KVO_DEV_BAD_COUNT; n = n < 0 ? 0 : k; }
    const int n_tok = n * B;
    const int64_t row0 = (int64_t)b * Hq + gk * r;      // the group's first output row
    WA st;
    {
        const bool v0 = gq < r, v1 = NR == 2 && gq + 8 < r;
        st.init(q + (row0 + (v0 ? gq : 0)) * D, q + (row0 + (v1 ? gq + 8 : 0)) * D, v0, v1, tq);
    }
    auto row_ptr = [&](const uint16_t* base, int tok) -> const uint16_t* {
        const int blk = tok / B;
        int sl = slot[(int64_t)bg * k + blk];
        if (sl < 0 || sl >= 2 * k) { bad |= KVO_DEV_BAD_SLOT; sl = 0; }
        return base + (((int64_t)bg * 2 * k + sl) * B + (tok - blk * B)) * D;
    };
    const int stride = S * ATT_WARPS * ATT_TILE;
    for (int tb = (sl_i * ATT_WARPS + warp) * ATT_TILE; tb < n_tok; tb += stride) {
        if (tb + stride < n_tok) {
            // lane l: token l & 15 of the warp's next tile, K rows for l < 16, V rows otherwise
            const int ntok = min(tb + stride + (lane & 15), n_tok - 1);
            const char* p = (const char*)row_ptr(lane < 16 ? bk : bv, ntok);
#pragma unroll
            for (int off = 0; off < D * 2; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
        }
        uint4 kf[2][CH];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint16_t* kp = row_ptr(bk, min(tb + 8 * nt + gq, n_tok - 1)) + 8 * tq;
#pragma unroll
            for (int s2 = 0; s2 < CH; ++s2) kf[nt][s2] = ldg16(kp + 32 * s2);
        }
        uint4 vf[4][CPT / 8];
#pragma unroll
        for (int vi = 0; vi < 4; ++vi) {
            const uint16_t* vp = row_ptr(bv, min(tb + 2 * tq + (vi & 1) + 8 * (vi >> 1), n_tok - 1)) + CPT * gq;
#pragma unroll
            for (int c = 0; c < CPT / 8; ++c) vf[vi][c] = ldg16(vp + 8 * c);
        }
        st.tile(kf, vf, tb, n_tok, scale_log2, tq);
    }
    if (bad && lane == 0) atomicOr(status, bad);
    st.to_smem(sm_m, sm_l, sm_o + warp * 8 * NR * D, warp, gq, tq);
    __syncthreads();
    // this CTA's part: unnormalised sum a and mass l relative to its maximum M (log2 domain)
    auto cta_part = [&](int row, int c, float& M, float& a, float& l) {
        M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w) M = fmaxf(M, sm_m[w][row]);
        a = 0.f; l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < ATT_WARPS; ++w) {
                const float sc = ex2f(sm_m[w][row] - M);
                a += sc * sm_o[w * 8 * NR * D + WA::state_idx(row, c)];
                l += sc * sm_l[w][row];
            }
        }
    };
    if (S > 1) {
        const int64_t pbase = ((int64_t)bg * S + sl_i) * r;
        for (int e = tid; e < r * D; e += ATT_WARPS * 32) {
            const int row = e / D, c = e - row * D;
            float M, a, l;
            cta_part(row, c, M, a, l);
            part_o[(pbase + row) * D + c] = a;
            if (c == 0) { part_ml[(pbase + row) * 2] = M; part_ml[(pbase + row) * 2 + 1] = l; }
        }
        // the same release / acquire ticket as the attention epilogue
        __syncthreads();
        if (tid == 0) {
            fence_acq_rel_gpu();
            const bool last = atomicAdd(&done[bg], 1u) + 1 == (uint32_t)S;
            if (last) fence_acq_rel_gpu();
            s_last = last;
        }
        __syncthreads();
        if (!s_last) return;
    }
    constexpr float kLog2e = 1.4426950408889634f;
    for (int e = tid; e < r * D; e += ATT_WARPS * 32) {
        const int row = e / D, c = e - row * D;
        float M, a, l;
        if (S == 1) {
            cta_part(row, c, M, a, l);
        } else {
            M = -INFINITY; a = 0.f; l = 0.f;
            for (int j = 0; j < S; ++j) {
                const int64_t pr = ((int64_t)bg * S + j) * r + row;
                const float mj = __ldcg(part_ml + pr * 2);
                if (mj == -INFINITY) continue;
                const float Mn = fmaxf(M, mj);
                const float so = ex2f(M - Mn), sn = ex2f(mj - Mn);
                l = l * so + __ldcg(part_ml + pr * 2 + 1) * sn;
                a = a * so + __ldcg(part_o + pr * D + c) * sn;
                M = Mn;
            }
        }
        // the prior part: normalised output and lse (natural log) -> mass 2^(lse*log2e - Mx)
        const int64_t orow = row0 + row;
        const float pl = prior_lse[orow] * kLog2e;
        const float Mx = fmaxf(pl, M);
        float o = 0.f, lse = -INFINITY;
        if (Mx != -INFINITY) {
            const float wp = pl == -INFINITY ? 0.f : ex2f(pl - Mx);
            const float wn = M == -INFINITY ? 0.f : ex2f(M - Mx);
            const float L = wp + wn * l;
            o = (wp * prior_o[orow * D + c] + wn * a) / L;
            lse = (Mx + lg2f(L)) * kLn2;
        }
        out_o[orow * D + c] = o;
        if (c == 0) out_lse[orow] = lse;
    }
    if (S > 1 && tid == 0) done[bg] = 0u;
}

// CTAs per group of attn_merge_part_kernel: enough for about four per SM, 1..MP_SPLIT_MAX
int merge_part_split(const Ctx& c) {
    return std::max(1, std::min(MP_SPLIT_MAX, (4 * std::max(1, c.n_sms)) / std::max(1, c.G)));
}

cudaError_t launch_attn_merge_part(const Ctx& c, int buf, const void* q, const int32_t* slot, const int32_t* cnt,
                                   const float* prior_o, const float* prior_lse, float* o, float* lse,
                                   cudaStream_t s) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.d));
    const int S = merge_part_split(c);
    if (S > 1 && (!c.mp_part_o || !c.mp_part_ml || !c.mp_done)) return cudaErrorInvalidValue;
    const dim3 grid(c.G, S);
#define KVO_MP(D_, NR_)                                                                                          \
    attn_merge_part_kernel<D_, NR_><<<grid, ATT_WARPS * 32, 0, s>>>((const uint16_t*)q, c.buf_k(buf), c.buf_v(buf), \
                                                                   slot, cnt, prior_o, prior_lse, o, lse,       \
                                                                   c.mp_part_o, c.mp_part_ml, c.mp_done, c.r,   \
                                                                   c.Hkv, c.k, c.B, scale_log2, c.status)
    if (c.d == 128) {
        if (c.r <= 8) KVO_MP(128, 1); else KVO_MP(128, 2);
    } else {
        if (c.r <= 8) KVO_MP(64, 1); else KVO_MP(64, 2);
    }
#undef KVO_MP
    return cudaGetLastError();
}

// --------------------------------------------------------------- merge_lse
__global__ void merge_lse_kernel(const float* __restrict__ o1, const float* __restrict__ lse1,
                                 const float* __restrict__ o2, const float* __restrict__ lse2, float* o, float* lse,
                                 int rows, int d) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= (int64_t)rows * d) return;
    const int64_t row = i / d;
    const float a = lse1[row], bb = lse2[row];
    const float M = fmaxf(a, bb);
    float out = 0.f, L = -INFINITY;
    if (M != -INFINITY) {
        const float l2e = 1.4426950408889634f;
        const float w1 = a == -INFINITY ? 0.f : ex2f((a - M) * l2e);
        const float w2 = bb == -INFINITY ? 0.f : ex2f((bb - M) * l2e);
        out = (w1 * o1[i] + w2 * o2[i]) / (w1 + w2);
        L = M + lg2f(w1 + w2) * kLn2;
    }
    o[i] = out;
    if (i % d == 0) lse[row] = L;
}

cudaError_t launch_merge_lse(const float* o1, const float* lse1, const float* o2, const float* lse2, float* o,
                             float* lse, int rows, int d, cudaStream_t s) {
    const int64_t n = (int64_t)rows * d;
    if (n == 0) return cudaSuccess;
    merge_lse_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(o1, lse1, o2, lse2, o, lse, rows, d);
    return cudaGetLastError();
}

}  // namespace kvo

// ---------------------------------------------------------------------------
// sparse_decode_attn_static: the attention kernel above, launched without a
// context and without allocating, for callers that cannot call cudaMalloc
// (their device memory belongs to another allocator, or their decode loop
// cannot afford the implicit synchronisation of cudaMalloc / cudaFree).
// Its work items, tickets and partial results
// live in one file-scope device array (kStaticAttnBytes, held by every GPU
// that loads the library until the process exits).  Host code cannot use the
// array's name as a device address, so the first call on each device looks
// the address up with cudaGetSymbolAddress (with that device current) and
// caches it.  Calls share the array: two calls that overlap on the GPU race.
// ---------------------------------------------------------------------------
#include <mutex>

namespace kvo {

constexpr size_t kStaticAttnBytes = size_t(24) << 20;
static __device__ __align__(256) unsigned char g_attn_static[kStaticAttnBytes];

__global__ void static_items_kernel(int4* __restrict__ items, int32_t* __restrict__ first,
                                    int32_t* __restrict__ count, int G, int sp_tiles, int w_tiles) {
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= G) return;
    const int sp_items = (sp_tiles + ATT_TILES_PER_ITEM - 1) / ATT_TILES_PER_ITEM;
    const int w_items = (w_tiles + ATT_TILES_PER_ITEM - 1) / ATT_TILES_PER_ITEM;
    const int base = g * (sp_items + w_items);
    first[g] = base;
    count[g] = sp_items + w_items;
    for (int i = 0; i < sp_items; ++i) {
        const int t = i * ATT_TILES_PER_ITEM;
        items[base + i] = make_int4(g, 0, t, min(ATT_TILES_PER_ITEM, sp_tiles - t));
    }
    for (int i = 0; i < w_items; ++i) {
        const int t = i * ATT_TILES_PER_ITEM;
        items[base + sp_items + i] = make_int4(g, 1, t, min(ATT_TILES_PER_ITEM, w_tiles - t));
    }
}

namespace {
std::mutex g_static_mu;
constexpr int kMaxDevices = 64;
unsigned char* g_static_addr[kMaxDevices] = {};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

}  // namespace kvo

extern "C" kvo_status sparse_decode_attn_static(const void* q, const void* k_buf, const void* v_buf,
                                                const int32_t* slot_of_true, const void* k_win, const void* v_win,
                                                float* o, float* lse, int32_t* status, int batch, int n_q_heads,
                                                int n_kv_heads, int head_dim, int block_size, int top_k,
                                                int window, int fuse_window_merge, kvo_stream_t stream) {
    using namespace kvo;
    auto bad = [](const char* m) { set_last_error(m); return KVO_ERR_INVALID; };
    if (batch < 1 || n_kv_heads < 1 || n_q_heads < n_kv_heads || n_q_heads % n_kv_heads)
        return bad("bad batch or head counts");
    const int r = n_q_heads / n_kv_heads;
    if (r > 16) return bad("n_q_heads / n_kv_heads must be <= 16");
    if (head_dim != 64 && head_dim != 128) return bad("head_dim must be 64 or 128");
    if (block_size < 1 || top_k < 1 || window < 0) return bad("need block_size >= 1, top_k >= 1, window >= 0");
    if (!q || !k_buf || !v_buf || !slot_of_true || !o || !lse) return bad("null pointer argument");
    if (window > 0 && (!k_win || !v_win)) return bad("window > 0 needs k_win and v_win");
    for (const void* p : {q, k_buf, v_buf, k_win, v_win})
        if ((uintptr_t)p % 16) return bad("bf16 inputs must be 16-byte aligned");
    const int G = batch * n_kv_heads;
    const int sp_tiles = (int)(((int64_t)top_k * block_size + ATT_TILE - 1) / ATT_TILE);
    const int w_tiles = (window + ATT_TILE - 1) / ATT_TILE;
    const int64_t per = (sp_tiles + ATT_TILES_PER_ITEM - 1) / ATT_TILES_PER_ITEM +
                        (w_tiles + ATT_TILES_PER_ITEM - 1) / ATT_TILES_PER_ITEM;
    const int64_t n_items = per * G;
    // layout: status word | tickets [G] | first [G] | count [G] | items | m,l | partial o
    const size_t off_done = 256;
    const size_t off_first = align256(off_done + 4 * (size_t)G);
    const size_t off_count = align256(off_first + 4 * (size_t)G);
    const size_t off_items = align256(off_count + 4 * (size_t)G);
    const size_t off_ml = align256(off_items + 16 * (size_t)n_items);
    const size_t off_o = align256(off_ml + 8 * (size_t)n_items * r);
    const size_t need = off_o + 4 * (size_t)n_items * r * head_dim;
    if (n_items > INT32_MAX || need > kStaticAttnBytes) {
        set_last_error(("sparse_decode_attn_static needs " + std::to_string(need) +
                        " bytes of static scratch; its capacity is " + std::to_string(kStaticAttnBytes) +
                        " bytes (reduce batch, KV heads, top_k * block_size or window)").c_str());
        return KVO_ERR_INVALID;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { set_last_error(cudaGetErrorString(e)); return KVO_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return bad("device ordinal beyond the static scratch table");
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_addr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_attn_static);
            if (e != cudaSuccess || !p) {
                set_last_error(("cudaGetSymbolAddress(static attention scratch): " +
                                std::string(cudaGetErrorString(e))).c_str());
                return KVO_ERR_CUDA;
            }
            g_static_addr[dev] = (unsigned char*)p;
        }
        base = g_static_addr[dev];
    }
    cudaStream_t s = (cudaStream_t)stream;
    int32_t* st = status ? status : (int32_t*)base;
    uint32_t* done = (uint32_t*)(base + off_done);
    int32_t* first = (int32_t*)(base + off_first);
    int32_t* count = (int32_t*)(base + off_count);
    int4* items = (int4*)(base + off_items);
    float* part_ml = (float*)(base + off_ml);
    float* part_o = (float*)(base + off_o);
    e = cudaMemsetAsync(done, 0, 4 * (size_t)G, s);
    if (e == cudaSuccess) {
        static_items_kernel<<<(G + 127) / 128, 128, 0, s>>>(items, first, count, G, sp_tiles, w_tiles);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
        const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)head_dim));
        const uint16_t* wk = window > 0 ? (const uint16_t*)k_win : nullptr;
        const uint16_t* wv = window > 0 ? (const uint16_t*)v_win : nullptr;
        const int fuse = fuse_window_merge ? 1 : 0;
#define KVO_ATT_STATIC(D_, NR_)                                                                                  \
        attn_kernel<D_, NR_><<<(unsigned)n_items, ATT_WARPS * 32, 0, s>>>(                                        \
            (const uint16_t*)q, nullptr, (const uint16_t*)k_buf, (const uint16_t*)v_buf, wk, wv, slot_of_true,  \
            items, first, count, part_o, part_ml, done, o, lse, nullptr, nullptr, fuse, batch, r, n_kv_heads,    \
            top_k, block_size, window, window, nullptr, nullptr, scale_log2, st)
        if (head_dim == 128) {
            if (r <= 8) KVO_ATT_STATIC(128, 1); else KVO_ATT_STATIC(128, 2);
        } else {
            if (r <= 8) KVO_ATT_STATIC(64, 1); else KVO_ATT_STATIC(64, 2);
        }
#undef KVO_ATT_STATIC
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) { set_last_error(cudaGetErrorString(e)); return KVO_ERR_CUDA; }
    return KVO_OK;
}
