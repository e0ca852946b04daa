// Growing the cache: one decode token per request and step.
//
// The recent window of "Scaling Attention Beyond GPUs for LLM Inference"
// (abstract: dense attention over the recent entries kept on the GPU, sparse
// attention over the salient offloaded ones) is a ring of W + B tokens per
// layer and (request, KV head).  A new token enters the ring; when the window
// holds W + B tokens its oldest block leaves it: the block's rows are written
// to the host cache and its K landmark ("DualDecoder: Accelerate Long Context
// LLM Inference by Predictive Prefetch", §4.1 / Fig. 8: static GPU-resident K
// landmarks) becomes candidate block C_b, so later selections can pick it.
//
// Token t of a group lives in ring slot t mod (W + B).  The window is tokens
// [C_b * B, len_b): between W and W + B - 1 of them.
#include "kvo_internal.cuh"

namespace kvo {

// ring slot (t mod Wcap) <- caller window row t - (len_b - W), for every window token t
__global__ void ring_fill_kernel(const uint16_t* __restrict__ wk, const uint16_t* __restrict__ wv,
                                 uint16_t* __restrict__ rk, uint16_t* __restrict__ rv,
                                 const int32_t* __restrict__ g_len, int W, int Wcap, int D) {
    const int bg = blockIdx.x;
    const int64_t t0 = (int64_t)g_len[bg] - W;
    const int words = D / 8;
    for (int i = threadIdx.x; i < W * words; i += blockDim.x) {
        const int j = i / words, w = i - j * words;
        const int slot = (int)((t0 + j) % Wcap);
        const int64_t src = ((int64_t)bg * W + j) * D + 8 * w;
        const int64_t dst = ((int64_t)bg * Wcap + slot) * D + 8 * w;
        *reinterpret_cast<uint4*>(rk + dst) = *reinterpret_cast<const uint4*>(wk + src);
        *reinterpret_cast<uint4*>(rv + dst) = *reinterpret_cast<const uint4*>(wv + src);
    }
}

cudaError_t launch_ring_fill(const Ctx& c, int layer, const uint16_t* k_win, const uint16_t* v_win, cudaStream_t s) {
    ring_fill_kernel<<<c.G, 256, 0, s>>>(k_win, v_win, c.ring_k[layer], c.ring_v[layer], c.g_len, c.W, c.Wcap, c.d);
    return cudaGetLastError();
}

// grid (G, L): write the new token; evict the oldest block when the window is full.
template <int D>
__global__ void __launch_bounds__(128)
append_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new, uint16_t* const* ring_k,
              uint16_t* const* ring_v, uint16_t* const* host_k, uint16_t* const* host_v, void* const* lm,
              const int64_t* __restrict__ g_off, const int32_t* __restrict__ g_C, const int32_t* __restrict__ g_len,
              int G, int B, int W, int Wcap, int Cmax) {
    constexpr int WORDS = D / 8;            // 16-byte words per row
    const int bg = blockIdx.x, l = blockIdx.y, tid = threadIdx.x;
    const int64_t t = g_len[bg];            // absolute index of the new token
    const int C = g_C[bg];
    uint16_t* rk = ring_k[l] + (int64_t)bg * Wcap * D;
    uint16_t* rv = ring_v[l] + (int64_t)bg * Wcap * D;
    const int64_t src = ((int64_t)l * G + bg) * D;      // k_new[l][b][g] == [l][bg]
    const int slot = (int)(t % Wcap);
    for (int w = tid; w < WORDS; w += blockDim.x) {
        *reinterpret_cast<uint4*>(rk + (int64_t)slot * D + 8 * w) = *reinterpret_cast<const uint4*>(k_new + src + 8 * w);
        *reinterpret_cast<uint4*>(rv + (int64_t)slot * D + 8 * w) = *reinterpret_cast<const uint4*>(v_new + src + 8 * w);
    }
    if (t + 1 - (int64_t)C * B != W + B) return;       // window not full yet
    // block C = tokens [C*B, C*B + B) leaves the window (its slots differ from the new token's)
    uint16_t* hk = host_k[l] + g_off[bg] + (int64_t)C * B * D;
    uint16_t* hv = host_v[l] + g_off[bg] + (int64_t)C * B * D;
    for (int i = tid; i < B * WORDS; i += blockDim.x) {
        const int row = i / WORDS, w = i - row * WORDS;
        const int s = (int)(((int64_t)C * B + row) % Wcap);
        *reinterpret_cast<uint4*>(hk + (int64_t)row * D + 8 * w) = *reinterpret_cast<const uint4*>(rk + (int64_t)s * D + 8 * w);
        *reinterpret_cast<uint4*>(hv + (int64_t)row * D + 8 * w) = *reinterpret_cast<const uint4*>(rv + (int64_t)s * D + 8 * w);
    }
    // landmark of block C: mean key in fp32 (chunk-major float4), or the bf16 key itself for B == 1
    if (B > 1) {
        float4* L4 = reinterpret_cast<float4*>(lm[l]) + (int64_t)bg * (D / 4) * Cmax;
        for (int c4 = tid; c4 < D / 4; c4 += blockDim.x) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            for (int row = 0; row < B; ++row) {
                const int s = (int)(((int64_t)C * B + row) % Wcap);
                const uint2 v = *reinterpret_cast<const uint2*>(rk + (int64_t)s * D + 4 * c4);
                a0 += bf16lo_to_f32(v.x); a1 += bf16hi_to_f32(v.x);
                a2 += bf16lo_to_f32(v.y); a3 += bf16hi_to_f32(v.y);
            }
            const float fb = (float)B;
            L4[(int64_t)c4 * Cmax + C] = make_float4(a0 / fb, a1 / fb, a2 / fb, a3 / fb);
        }
    } else {
        uint4* L8 = reinterpret_cast<uint4*>(lm[l]) + (int64_t)bg * WORDS * Cmax;
        const int s = (int)(((int64_t)C) % Wcap);
        for (int w = tid; w < WORDS; w += blockDim.x)
            L8[(int64_t)w * Cmax + C] = *reinterpret_cast<const uint4*>(rk + (int64_t)s * D + 8 * w);
    }
}

// one thread per group: advance the length, the candidate count and the window
__global__ void append_commit_kernel(int32_t* __restrict__ g_C, int32_t* __restrict__ g_len,
                                     int32_t* __restrict__ g_wstart, int32_t* __restrict__ g_wlen, int G, int B,
                                     int W, int Wcap) {
    const int bg = blockIdx.x * blockDim.x + threadIdx.x;
    if (bg >= G) return;
    const int len = g_len[bg] + 1;
    int C = g_C[bg];
    if (len - C * B == W + B) ++C;
    g_len[bg] = len;
    g_C[bg] = C;
    g_wstart[bg] = (int)(((int64_t)C * B) % Wcap);
    g_wlen[bg] = len - C * B;
}

cudaError_t launch_append(const Ctx& c, const void* k_new, const void* v_new, cudaStream_t s) {
    dim3 grid(c.G, c.L);
    if (c.d == 128)
        append_kernel<128><<<grid, 128, 0, s>>>((const uint16_t*)k_new, (const uint16_t*)v_new, c.d_ring_k,
                                                c.d_ring_v, c.d_host_k, c.d_host_v, c.d_lm, c.g_off, c.g_C, c.g_len,
                                                c.G, c.B, c.W, c.Wcap, c.Cmax);
    else
        append_kernel<64><<<grid, 128, 0, s>>>((const uint16_t*)k_new, (const uint16_t*)v_new, c.d_ring_k,
                                               c.d_ring_v, c.d_host_k, c.d_host_v, c.d_lm, c.g_off, c.g_C, c.g_len,
                                               c.G, c.B, c.W, c.Wcap, c.Cmax);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    append_commit_kernel<<<(c.G + 127) / 128, 128, 0, s>>>(c.g_C, c.g_len, c.g_wstart, c.g_wlen, c.G, c.B, c.W,
                                                           c.Wcap);
    return cudaGetLastError();
}

}  // namespace kvo
