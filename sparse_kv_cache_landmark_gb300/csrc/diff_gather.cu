// Predicted-vs-needed diff, run coalescing and the host -> HBM gather.
//
// "DualDecoder: Accelerate Long Context LLM Inference by Predictive Prefetch",
// §5.2 / Fig. 10 / Fig. 18: entries of the true retrieval index that the
// prediction missed are fetched on an urgent stream before attention;
// §5.4 / Fig. 11: a two-layer ping-pong sparse KV buffer; Fig. 19: contiguous
// block prefetch over the host link.  "PulseInfer and the I/O Problem Behind
// Long-Context Decoding", §2: a gather-scatter engine that coalesces
// fragmented transfers.
//
// Ping-pong half layout (HBM): [G][2k][B][d] bf16 for K and for V; slots
// [0, k) hold the prefetched prediction in list order, slots [k, 2k) the
// urgent misses in list order.  A run of n adjacent block ids is one
// contiguous range of n*B*d bf16 on both the host and the device side.
#include <algorithm>

#include "kvo_internal.cuh"

namespace kvo {

// ------------------------------------------------------------------- diff
__global__ void __launch_bounds__(256)
index_diff_kernel(const int32_t* __restrict__ T, const int32_t* __restrict__ P, int32_t* __restrict__ M,
                  int32_t* __restrict__ M_cnt, int32_t* __restrict__ slot, const int32_t* __restrict__ g_C, int k,
                  int32_t* __restrict__ status) {
    extern __shared__ int32_t p_s[];           // prediction of the group, k entries
    __shared__ uint32_t warp_sums[32];
    const int bg = blockIdx.x, tid = threadIdx.x;
    const int C = g_C[bg];
    const int32_t* Tg = T + (int64_t)bg * k;
    int bad = 0;
    if (P) {
        const int32_t* Pg = P + (int64_t)bg * k;
        for (int i = tid; i < k; i += blockDim.x) {
            const int32_t x = Pg[i];
            p_s[i] = x;
            if (x < 0 || x >= C) bad |= KVO_DEV_BAD_BLOCK_ID;
            if (i > 0 && Pg[i - 1] >= x) bad |= KVO_DEV_UNSORTED;
        }
    }
    __syncthreads();
    uint32_t n_miss = 0;
    for (int base = 0; base < k; base += blockDim.x) {
        const int i = base + tid;
        const bool valid = i < k;
        const int32_t t = valid ? Tg[i] : 0;
        if (valid && (t < 0 || t >= C)) bad |= KVO_DEV_BAD_BLOCK_ID;
        if (valid && i > 0 && Tg[i - 1] >= t) bad |= KVO_DEV_UNSORTED;
        int pos = -1;
        if (valid && P) {
            int lo = 0, hi = k - 1;
            while (lo <= hi) {
                const int mid = (lo + hi) >> 1;
                const int32_t v = p_s[mid];
                if (v == t) { pos = mid; break; }
                if (v < t) lo = mid + 1; else hi = mid - 1;
            }
        }
        const bool miss = valid && pos < 0;
        uint32_t total;
        const uint32_t excl = block_exclusive_scan(miss ? 1u : 0u, warp_sums, &total);
        if (miss) {
            M[(int64_t)bg * k + n_miss + excl] = t;
            slot[(int64_t)bg * k + i] = k + (int32_t)(n_miss + excl);
        } else if (valid) {
            slot[(int64_t)bg * k + i] = pos;
        }
        n_miss += total;
    }
    if (tid == 0) M_cnt[bg] = (int32_t)n_miss;
    if (bad) atomicOr(status, bad);
}

cudaError_t launch_index_diff(const Ctx& c, const int32_t* idx_true, const int32_t* idx_pred, int32_t* miss,
                              int32_t* miss_cnt, int32_t* slot, cudaStream_t s) {
    const size_t smem = idx_pred ? (size_t)c.k * sizeof(int32_t) : 0;
    index_diff_kernel<<<c.G, 256, smem, s>>>(idx_true, idx_pred, miss, miss_cnt, slot, c.g_C, c.k, c.status);
    return cudaGetLastError();
}

// --------------------------------------------------------------- coalesce
// runs[G][k] int4 = {first block, n blocks, first slot, 0}; nruns[G].
__global__ void __launch_bounds__(256)
coalesce_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int slot_base,
                int4* __restrict__ runs, int32_t* __restrict__ nruns, const int32_t* __restrict__ g_C, int k,
                int32_t* __restrict__ status) {
    __shared__ uint32_t warp_sums[32];
    const int bg = blockIdx.x, tid = threadIdx.x;
    const int C = g_C[bg];
    int n = cnt ? cnt[bg] : k;
    int bad = 0;
    if (n < 0 || n > k) { bad |= KVO_DEV_BAD_COUNT; n = n < 0 ? 0 : k; }
    const int32_t* S = idx + (int64_t)bg * k;
    int4* R = runs + (int64_t)bg * k;
    uint32_t n_start = 0, n_end = 0;
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + tid;
        const bool valid = i < n;
        const int32_t x = valid ? S[i] : 0;
        if (valid && (x < 0 || x >= C)) bad |= KVO_DEV_BAD_BLOCK_ID;
        const bool start = valid && (i == 0 || S[i - 1] + 1 != x);
        const bool end = valid && (i == n - 1 || S[i + 1] != x + 1);
        uint32_t ts, te;
        const uint32_t es = block_exclusive_scan(start ? 1u : 0u, warp_sums, &ts);
        const uint32_t ee = block_exclusive_scan(end ? 1u : 0u, warp_sums, &te);
        if (start) { R[n_start + es].x = x; R[n_start + es].y = i; R[n_start + es].z = slot_base + i; }
        if (end) R[n_end + ee].w = i;
        n_start += ts;
        n_end += te;
    }
    __syncthreads();
    for (int j = tid; j < (int)n_start; j += blockDim.x) {
        int4 v = R[j];
        v.y = v.w - v.y + 1;
        v.w = 0;
        R[j] = v;
    }
    if (tid == 0) nruns[bg] = (int32_t)n_start;
    if (bad) atomicOr(status, bad);
}

cudaError_t launch_coalesce(const Ctx& c, const int32_t* idx, const int32_t* cnt, int slot_base, int32_t* runs,
                            int32_t* nruns, cudaStream_t s) {
    coalesce_kernel<<<c.G, 256, 0, s>>>(idx, cnt, slot_base, (int4*)runs, nruns, c.g_C, c.k, c.status);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ gather
// One warp per run (grid-stride over the G*k run slots).  The host cache is
// read in place through its device mapping with 16-byte loads, UNROLL loads
// of K and of V in flight per lane, and written to the ping-pong half with
// coalesced 16-byte stores.
template <int UNROLL>
__global__ void __launch_bounds__(GATHER_THREADS)
gather_kernel(const uint16_t* __restrict__ kh, const uint16_t* __restrict__ vh, const int64_t* __restrict__ g_off,
              const int32_t* __restrict__ g_C, const int4* __restrict__ runs, const int32_t* __restrict__ nruns,
              uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, int G, int k, int B, int D,
              int32_t* __restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = (int64_t)G * k;
    const int64_t blk_elems = (int64_t)B * D;
    for (int64_t e = warp; e < total; e += n_warps) {
        const int bg = (int)(e / k);
        const int ri = (int)(e - (int64_t)bg * k);
        if (ri >= nruns[bg]) continue;
        const int4 run = runs[e];
        if (run.x < 0 || run.y < 1 || run.x + run.y > g_C[bg] || run.z < 0 || run.z + run.y > 2 * k) {
            if (lane == 0) atomicOr(status, KVO_DEV_BAD_SLOT);
            continue;
        }
        const int64_t src = g_off[bg] + (int64_t)run.x * blk_elems;
        const int64_t dst = ((int64_t)bg * 2 * k + run.z) * blk_elems;
        const int64_t n16 = (int64_t)run.y * blk_elems / 8;
        const uint4* sk = reinterpret_cast<const uint4*>(kh + src);
        const uint4* sv = reinterpret_cast<const uint4*>(vh + src);
        uint4* tk = reinterpret_cast<uint4*>(dk + dst);
        uint4* tv = reinterpret_cast<uint4*>(dv + dst);
        for (int64_t i0 = lane; i0 < n16; i0 += 32 * UNROLL) {
            uint4 a[UNROLL], b[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t i = i0 + 32 * u;
                if (i < n16) { a[u] = sk[i]; b[u] = sv[i]; }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t i = i0 + 32 * u;
                if (i < n16) { tk[i] = a[u]; tv[i] = b[u]; }
            }
        }
    }
}

// Flat variant: the index list itself is the copy plan.  Entry j of group bg
// (block idx[bg][j], j < cnt[bg]) goes to slot slot_base + j, so a run of
// adjacent block ids is one contiguous source range and one contiguous
// destination range.  Persistent warps walk chunks of 32*U 16-byte words of
// one group's entry stream (K and V): no per-run dependency chain, and a
// warp's metadata loads hit one or two cache lines.  With `compact` every CTA
// first builds, in shared memory, the prefix over the groups of their chunk
// counts (listed entries x words per block, rounded up to chunks), so the warps
// stride over the listed chunks only -- a short miss list costs a short walk --
// and find a chunk's group by binary search; without it (full lists, or more
// groups than the prefix may hold) the warps stride over k entries' chunks of
// every group.
// The launch may reserve shared memory it never uses so that each gather CTA
// has its SM to itself: the other kernels then never queue their HBM loads
// behind zero-copy loads waiting on the host link in the same SM's load/store
// pipeline.  With a slot list (dslot) entry j goes to slot dslot[bg][j]
// instead; kv_mask bit 0 copies K, bit 1 copies V (V alone where the keys are
// rebuilt on the GPU).
template <int U, bool POW2>
__global__ void __launch_bounds__(1024)
gather_flat_kernel(const uint16_t* __restrict__ kh, const uint16_t* __restrict__ vh,
                   const int64_t* __restrict__ g_off, const int32_t* __restrict__ g_C,
                   const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int slot_base,
                   const int32_t* __restrict__ dslot,
                   uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, int G, int k, int B, int D, int words_log2,
                   int kv_mask, bool compact, int32_t* __restrict__ status) {
    // a kernel launched as this one's programmatic dependent may start as soon
    // as every CTA of this grid is resident (it waits for this grid's
    // completion before it reads what this grid writes)
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr uint32_t CHUNK = 32 * U;                       // words per warp iteration
    extern __shared__ uint32_t s_pre[];                      // [G + 1] chunk prefix (compact)
    __shared__ uint32_t s_wsum[32];
    const uint32_t words = (uint32_t)B * D / 8;             // 16-byte words per block
    const uint32_t per_group = ((uint32_t)k * words + CHUNK - 1) / CHUNK;   // chunks per group
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    int bad = 0;
    int64_t total = (int64_t)G * per_group;
    if (compact) {
        // block-wide exclusive scan: thread t owns groups [t*per, t*per + per)
        const int nt = blockDim.x, t = threadIdx.x, per = (G + nt - 1) / nt;
        const int g0 = min(t * per, G), g1 = min(g0 + per, G);
        auto chunks_of = [&](int g, int& flag) -> uint32_t {
            int n = cnt ? __ldg(cnt + g) : k;
            if (n < 0 || n > k) { flag |= KVO_DEV_BAD_COUNT; n = n < 0 ? 0 : k; }
            return ((uint32_t)n * words + CHUNK - 1) / CHUNK;
        };
        int flag = 0;
        uint32_t own = 0;
        for (int g = g0; g < g1; ++g) own += chunks_of(g, flag);
        uint32_t inc = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) s_wsum[t >> 5] = inc;
        __syncthreads();
        if (t < 32) {
            uint32_t x = t < (nt >> 5) ? s_wsum[t] : 0u, xi = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, xi, o);
                if (lane >= o) xi += y;
            }
            s_wsum[t] = xi - x;                              // exclusive prefix of the warp sums
            if (t == 31) s_pre[G] = xi;                      // all chunks
        }
        __syncthreads();
        uint32_t run = s_wsum[t >> 5] + inc - own;
        int unused = 0;
        for (int g = g0; g < g1; ++g) { s_pre[g] = run; run += chunks_of(g, unused); }
        if (blockIdx.x == 0) bad |= flag;                   // counts are reported once
        __syncthreads();
        total = s_pre[G];
    }
    for (int64_t ch = warp; ch < total; ch += n_warps) {
        int bg;
        uint32_t c0;
        if (compact) {
            // the last group whose first chunk is <= ch (groups without chunks share their successor's start)
            int lo = 0, hi = G - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_pre[mid] <= (uint32_t)ch) lo = mid; else hi = mid - 1;
            }
            bg = lo;
            c0 = ((uint32_t)ch - s_pre[bg]) * CHUNK;
        } else {
            bg = (int)(ch / per_group);
            c0 = (uint32_t)(ch - (int64_t)bg * per_group) * CHUNK;
        }
        int n = cnt ? cnt[bg] : k;
        if (n < 0 || n > k) { if (!compact) bad |= KVO_DEV_BAD_COUNT; n = n < 0 ? 0 : k; }
        const uint32_t lim = (uint32_t)n * words;
        if (c0 >= lim) continue;
        const int C = g_C[bg];
        const int64_t src0 = g_off[bg];
        const int32_t* ig = idx + (int64_t)bg * k;
        const int32_t* sg = dslot ? dslot + (int64_t)bg * k : nullptr;
        uint4 a[U], b[U];
        int64_t to[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t i = c0 + u * 32 + lane;
            ok[u] = false;
            if (i < lim) {
                const uint32_t j = POW2 ? (i >> words_log2) : (i / words);
                const uint32_t w = i - j * words;
                const int32_t blk = __ldg(ig + j);
                // destination: slot slot_base + j, or the entry's own slot when a slot list is given
                const int32_t sl = sg ? __ldg(sg + j) : slot_base + (int32_t)j;
                if (blk >= 0 && blk < C && sl >= 0 && sl < 2 * k) {
                    const int64_t off = (int64_t)blk * B * D + 8 * (int64_t)w;
                    if (kv_mask & 1) a[u] = *reinterpret_cast<const uint4*>(kh + src0 + off);
                    if (kv_mask & 2) b[u] = *reinterpret_cast<const uint4*>(vh + src0 + off);
                    to[u] = ((int64_t)bg * 2 * k + sl) * B * D + 8 * (int64_t)w;
                    ok[u] = true;
                } else {
                    bad |= (blk >= 0 && blk < C) ? KVO_DEV_BAD_SLOT : KVO_DEV_BAD_BLOCK_ID;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (ok[u]) {
                if (kv_mask & 1) *reinterpret_cast<uint4*>(dk + to[u]) = a[u];
                if (kv_mask & 2) *reinterpret_cast<uint4*>(dv + to[u]) = b[u];
            }
    }
    if (bad) atomicOr(status, bad);
}

// Largest group count whose chunk prefix the flat gather keeps in shared memory.
constexpr int FLAT_PREFIX_MAX_G = 16384;

cudaError_t launch_gather_flat(const Ctx& c, int layer, int buf, const int32_t* idx, const int32_t* cnt, int slot_base,
                               cudaStream_t s, const int32_t* dslot, int kv_mask, bool alone) {
    const uint32_t words = (uint32_t)c.B * c.d / 8;
    int lg = -1;
    if ((words & (words - 1)) == 0) { lg = 0; while ((1u << lg) < words) ++lg; }
    // `alone`: nothing else runs beside this copy, so it takes every SM (one
    // 1024-thread CTA each, no reservation) to cut the latency of small lists
    const int ctas = alone ? c.n_sms : (c.gather_ctas > 0 ? c.gather_ctas : 2 * 152);
    const int th = alone ? 1024 : c.gather_threads;
    // Lists with counts walk the listed chunks through the prefix (G + 1 words,
    // no 32-bit overflow); full lists (no counts) have no empty chunk to skip
    // and stride over k entries per group without the per-chunk group search.
    const int U = c.gather_unroll >= 2 ? 2 : 1;
    const int64_t all_chunks = (int64_t)c.G * (((int64_t)c.k * words + 32 * U - 1) / (32 * U));
    const bool compact = cnt && c.G <= FLAT_PREFIX_MAX_G && all_chunks < (int64_t)1 << 31;
    const size_t pre = compact ? sizeof(uint32_t) * (c.G + 1) : 0;
    const size_t smem = std::max(alone ? (size_t)0 : (size_t)c.gather_reserve_smem, pre);
#define KVO_FLAT(U_, P_)                                                                                          \
    gather_flat_kernel<U_, P_><<<ctas, th, smem, s>>>(c.k_host[layer], c.v_host[layer], c.g_off, c.g_C, idx, cnt, \
                                                      slot_base, dslot, c.buf_k(buf), c.buf_v(buf), c.G, c.k,     \
                                                      c.B, c.d, lg, kv_mask, compact, c.status)
    if (lg >= 0) { if (U == 2) KVO_FLAT(2, true); else KVO_FLAT(1, true); }
    else { if (U == 2) KVO_FLAT(2, false); else KVO_FLAT(1, false); }
#undef KVO_FLAT
    return cudaGetLastError();
}

cudaError_t prepare_gather_flat() {
    const int mx = 227 * 1024 - 32 * (int)sizeof(uint32_t);     // less the warp-sum table
    cudaError_t e = cudaFuncSetAttribute(gather_flat_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gather_flat_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gather_flat_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gather_flat_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    return e;
}

int gather_default_ctas(const Ctx& c) {
    return c.gather_ctas > 0 ? c.gather_ctas : 2 * 152;
}

__global__ void status_or_kernel(int32_t* status, int bits) { atomicOr(status, bits); }

// Copy engine: the run list is read back to the host (the stream is
// synchronised for it), then every run becomes one cudaMemcpyAsync of K and
// one of V from the pinned host cache into the buffer's slots, on the stream.
// No SM takes part in moving the bytes; the host issues one call per copy.
// A run outside the group's blocks or the buffer's slots is skipped and
// reported in the device status word.
static cudaError_t gather_copy_engine(const Ctx& c, int layer, int buf, const int32_t* runs, const int32_t* nruns,
                                      cudaStream_t s) {
    if (!c.h_runs || !c.h_nruns || c.h_off.size() != (size_t)c.G) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemcpyAsync(c.h_nruns, nruns, sizeof(int32_t) * c.G, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(c.h_runs, runs, sizeof(int32_t) * 4 * (size_t)c.G * c.k, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    const int64_t blk = (int64_t)c.B * c.d;
    bool bad = false;
    for (int g = 0; g < c.G; ++g) {
        const int n = std::min(std::max(c.h_nruns[g], 0), c.k);
        for (int j = 0; j < n; ++j) {
            const int32_t* r = c.h_runs + 4 * ((int64_t)g * c.k + j);
            const int32_t x = r[0], nb = r[1], sl = r[2];
            if (x < 0 || nb < 1 || (int64_t)x + nb > c.h_Ccap[g] || sl < 0 || sl + nb > 2 * c.k) {
                bad = true;
                continue;
            }
            const int64_t src = c.h_off[g] + x * blk, dst = ((int64_t)g * 2 * c.k + sl) * blk;
            const size_t bytes = (size_t)nb * blk * sizeof(uint16_t);
            e = cudaMemcpyAsync(c.buf_k(buf) + dst, c.k_host[layer] + src, bytes, cudaMemcpyDefault, s);
            if (e == cudaSuccess) e = cudaMemcpyAsync(c.buf_v(buf) + dst, c.v_host[layer] + src, bytes, cudaMemcpyDefault, s);
            if (e != cudaSuccess) return e;
        }
    }
    if (bad) {
        status_or_kernel<<<1, 1, 0, s>>>(c.status, KVO_DEV_BAD_SLOT);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

cudaError_t launch_gather(const Ctx& c, int layer, int buf, const int32_t* runs, const int32_t* nruns,
                          cudaStream_t s) {
    if (c.gather_engine == 1) return launch_gather_tma(c, layer, buf, runs, nruns, s);
    if (c.gather_engine == 4) return gather_copy_engine(c, layer, buf, runs, nruns, s);
    const int ctas = gather_default_ctas(c), th = c.gather_threads;
#define KVO_GATHER(U_)                                                                                          \
    gather_kernel<U_><<<ctas, th, 0, s>>>(c.k_host[layer], c.v_host[layer], c.g_off, c.g_C, (const int4*)runs, \
                                          nruns, c.buf_k(buf), c.buf_v(buf), c.G, c.k, c.B, c.d, c.status)
    if (c.gather_unroll >= 4) KVO_GATHER(4);
    else if (c.gather_unroll == 2) KVO_GATHER(2);
    else KVO_GATHER(1);
#undef KVO_GATHER
    return cudaGetLastError();
}

}  // namespace kvo
