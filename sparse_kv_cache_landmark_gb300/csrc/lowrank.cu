// Low-rank key reconstruction for missed blocks ("DualDecoder: Accelerate Long
// Context LLM Inference by Predictive Prefetch", §5.3: for some layers the keys
// of missed entries are rebuilt on the GPU from a GPU-resident low-rank key
// cache instead of being fetched; only their values cross the host link).
//
// A layer's keys are given as rank-R factors: per (request, KV head) bf16
// coefficients a[t][R] for every token and a bf16 basis e[R][d].  The key row
// of token t is bf16( sum over j ascending of a[t][j] * e[j][c] ), each product
// and each partial sum rounded to fp32 (no fused multiply-add), rounded to bf16
// to nearest-even at the end -- the definition of the synthetic low-rank keys,
// so the rebuilt rows equal the host rows bit for bit.
#include <cuda_bf16.h>

#include "kvo_internal.cuh"

namespace kvo {

constexpr int LR_THREADS = 256;
constexpr int LR_ROWS = 64;        // token rows per CTA

// Grid (group, row chunk): CTA y rebuilds the chunks y, y + gridDim.y, ... of
// LR_ROWS rows of the group's listed blocks (entry j -> slot slot_base + j, or
// dslot[j]; row j*B + i is token i of block j) into the K buffer; CTAs whose
// first chunk lies past the list's rows exit at once.  A warp owns one row at a time; lane l holds channels
// CPL*l .. CPL*l + CPL-1.
template <int D>
__global__ void __launch_bounds__(LR_THREADS)
lowrank_k_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int slot_base,
                 const int32_t* __restrict__ dslot, const uint16_t* __restrict__ coef,
                 const uint16_t* __restrict__ basis, const int64_t* __restrict__ g_off,
                 const int32_t* __restrict__ g_C, uint16_t* __restrict__ dk, int k, int B, int R,
                 int32_t* __restrict__ status) {
    constexpr int CPL = D / 32;                    // channels per lane
    extern __shared__ float e_s[];                 // [R][D] fp32 basis
    const int bg = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int n = cnt ? cnt[bg] : k;
    int bad = 0;
    if (n < 0 || n > k) { bad |= KVO_DEV_BAD_COUNT; n = n < 0 ? 0 : k; }
    const int nrows = n * B;
    if ((int64_t)blockIdx.y * LR_ROWS >= nrows) {
        if (bad && tid == 0 && blockIdx.y == 0) atomicOr(status, bad);
        return;
    }
    const uint16_t* eb = basis + (int64_t)bg * R * D;
    for (int i = tid; i < R * D; i += blockDim.x)
        e_s[i] = __uint_as_float((uint32_t)eb[i] << 16);
    __syncthreads();
    const int C = g_C[bg];
    const int64_t row0 = g_off[bg] / D;            // the group's first token row
    for (int64_t rr = (int64_t)blockIdx.y * LR_ROWS + warp; rr < nrows;
         rr += ((rr % LR_ROWS) + LR_THREADS / 32 >= LR_ROWS) ? (int64_t)(gridDim.y - 1) * LR_ROWS + LR_THREADS / 32
                                                             : LR_THREADS / 32) {
        const int j = (int)(rr / B), i = (int)(rr - (int64_t)j * B);
        const int32_t x = __ldg(idx + (int64_t)bg * k + j);
        const int32_t s = dslot ? __ldg(dslot + (int64_t)bg * k + j) : slot_base + j;
        if (x < 0 || x >= C || s < 0 || s >= 2 * k) {
            bad |= (x < 0 || x >= C) ? KVO_DEV_BAD_BLOCK_ID : KVO_DEV_BAD_SLOT;
            continue;
        }
        const uint16_t* ar = coef + (row0 + (int64_t)x * B + i) * R;
        // lane l holds coefficients l and l + 32
        const float a_lo = lane < R ? __uint_as_float((uint32_t)ar[lane] << 16) : 0.f;
        const float a_hi = lane + 32 < R ? __uint_as_float((uint32_t)ar[lane + 32] << 16) : 0.f;
        float acc[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
        for (int jj = 0; jj < R; ++jj) {
            const float a = __shfl_sync(0xffffffffu, jj < 32 ? a_lo : a_hi, jj & 31);
            const float* er = e_s + jj * D + CPL * lane;
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = __fadd_rn(acc[c], __fmul_rn(a, er[c]));
        }
        uint16_t* out = dk + (((int64_t)bg * 2 * k + s) * B + i) * D + CPL * lane;
#pragma unroll
        for (int c = 0; c < CPL; c += 2) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(acc[c], acc[c + 1]);
            *reinterpret_cast<__nv_bfloat162*>(out + c) = v;
        }
    }
    if (bad && lane == 0) atomicOr(status, bad);
}

cudaError_t prepare_lowrank() {
    const int mx = 64 * 128 * 4;
    cudaError_t e = cudaFuncSetAttribute(lowrank_k_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lowrank_k_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    return e;
}

cudaError_t launch_lowrank_k(const Ctx& c, int layer, int buf, const int32_t* idx, const int32_t* cnt, int slot_base,
                             const int32_t* dslot, cudaStream_t s) {
    const int R = c.lr_rank[layer];
    const size_t smem = sizeof(float) * R * c.d;
    const int64_t chunks = ((int64_t)c.k * c.B + LR_ROWS - 1) / LR_ROWS;
    const dim3 grid(c.G, (unsigned)std::min<int64_t>(chunks, 65535));
    if (c.d == 128)
        lowrank_k_kernel<128><<<grid, LR_THREADS, smem, s>>>(idx, cnt, slot_base, dslot, c.lr_coef[layer],
                                                            c.lr_basis[layer], c.g_off, c.g_C, c.buf_k(buf), c.k,
                                                            c.B, R, c.status);
    else
        lowrank_k_kernel<64><<<grid, LR_THREADS, smem, s>>>(idx, cnt, slot_base, dslot, c.lr_coef[layer],
                                                           c.lr_basis[layer], c.g_off, c.g_C, c.buf_k(buf), c.k,
                                                           c.B, R, c.status);
    return cudaGetLastError();
}

}  // namespace kvo
