// K landmarks and retrieval-index selection.
//
// "DualDecoder: Accelerate Long Context LLM Inference by Predictive Prefetch",
// §4.1 / Fig. 6 / Fig. 8: the retrieval index of a decode step is computed from
// a (true or speculative) token and static GPU-resident K landmarks.  Landmark
// of block j = mean key of its B tokens (fp32; for B == 1 the bf16 key itself).
// Score of block j for KV head g = sum over the group's query heads of q_h . L_j.
// The index is the exact top-k, ascending, ties to the lower block id.
//
// Layout of the landmarks of one layer (HBM, resident):
//   B > 1 : float4 [G][d/4][Cmax]   (channel-chunk major: thread j reads row j
//           one 16-byte chunk at a time, a warp reads 512 contiguous bytes)
//   B == 1: uint4  [G][d/8][Cmax]   (8 bf16 per chunk)
// Selection is one kernel: CTAs score chunks of landmark rows of one group,
// write order-preserving uint32 keys and a histogram of their top 8 bits; the
// last CTA of a group (atomic ticket) finishes an MSB radix select (up to 4
// passes of 8 bits, ending early on a bin whose keys are all wanted) on
// the L2-resident keys and compacts the winners in ascending id order.  Where
// a group's CTAs fit one thread-block cluster, select_cluster_kernel (below)
// can run the radix select on all of them instead.
#include <algorithm>

#include "kvo_internal.cuh"
#include "resident_assign.cuh"
#include "tma_ptx.cuh"

namespace kvo {

// ------------------------------------------------------------- landmarks
template <int D>
__global__ void landmark_mean_kernel(const uint16_t* __restrict__ kh, const int64_t* __restrict__ g_off,
                                     const int32_t* __restrict__ g_C, float4* __restrict__ lm, int Cmax, int B) {
    const int bg = blockIdx.y;
    const int warps = blockDim.x >> 5;
    const int j = blockIdx.x * warps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int C = g_C[bg];
    if (j >= C || lane >= D / 4) return;
    const uint16_t* src = kh + g_off[bg] + (int64_t)j * B * D + 4 * lane;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int t = 0; t < B; ++t) {
        uint2 w = *reinterpret_cast<const uint2*>(src + (int64_t)t * D);
        s0 += bf16lo_to_f32(w.x); s1 += bf16hi_to_f32(w.x);
        s2 += bf16lo_to_f32(w.y); s3 += bf16hi_to_f32(w.y);
    }
    const float fb = (float)B;
    lm[((int64_t)bg * (D / 4) + lane) * Cmax + j] = make_float4(s0 / fb, s1 / fb, s2 / fb, s3 / fb);
}

template <int D>
__global__ void landmark_copy_kernel(const uint16_t* __restrict__ kh, const int64_t* __restrict__ g_off,
                                     const int32_t* __restrict__ g_C, uint4* __restrict__ lm, int Cmax) {
    constexpr int LPT = D / 8;              // lanes per token
    constexpr int TPW = 32 / LPT;           // tokens per warp
    const int bg = blockIdx.y;
    const int warps = blockDim.x >> 5;
    const int lane = threadIdx.x & 31;
    const int j = (blockIdx.x * warps + (threadIdx.x >> 5)) * TPW + lane / LPT;
    const int c8 = lane % LPT;
    if (j >= g_C[bg]) return;
    const uint4 v = *reinterpret_cast<const uint4*>(kh + g_off[bg] + (int64_t)j * D + 8 * c8);
    lm[((int64_t)bg * LPT + c8) * Cmax + j] = v;
}

cudaError_t launch_landmarks(const Ctx& c, int layer, cudaStream_t s) {
    const int threads = 256, warps = threads / 32;
    if (c.B > 1) {
        dim3 grid((c.Cmax + warps - 1) / warps, c.G);
        if (c.d == 128)
            landmark_mean_kernel<128><<<grid, threads, 0, s>>>(c.k_host[layer], c.g_off, c.g_C,
                                                               (float4*)c.lm[layer], c.Cmax, c.B);
        else
            landmark_mean_kernel<64><<<grid, threads, 0, s>>>(c.k_host[layer], c.g_off, c.g_C,
                                                              (float4*)c.lm[layer], c.Cmax, c.B);
    } else {
        const int tpw = 32 / (c.d / 8);
        dim3 grid((c.Cmax + warps * tpw - 1) / (warps * tpw), c.G);
        if (c.d == 128)
            landmark_copy_kernel<128><<<grid, threads, 0, s>>>(c.k_host[layer], c.g_off, c.g_C,
                                                               (uint4*)c.lm[layer], c.Cmax);
        else
            landmark_copy_kernel<64><<<grid, threads, 0, s>>>(c.k_host[layer], c.g_off, c.g_C,
                                                              (uint4*)c.lm[layer], c.Cmax);
    }
    return cudaGetLastError();
}

// logical copy [G][Cmax][d] for inspection
template <typename T, int CH>
__global__ void landmark_unpermute_kernel(const T* __restrict__ lm, T* __restrict__ out, int Cmax, int nchunk) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;   // over G*Cmax*nchunk
    const int64_t per_g = (int64_t)Cmax * nchunk;
    const int64_t total = per_g * gridDim.y;
    const int bg = blockIdx.y;
    if (i >= per_g) return;
    (void)total;
    const int j = (int)(i / nchunk), ch = (int)(i % nchunk);
    out[((int64_t)bg * Cmax + j) * nchunk + ch] = lm[((int64_t)bg * nchunk + ch) * Cmax + j];
}

cudaError_t copy_landmarks_logical(const Ctx& c, int layer, void* dst, cudaStream_t s) {
    const int64_t per_g = (int64_t)c.Cmax * (c.B > 1 ? c.d / 4 : c.d / 8);
    dim3 grid((unsigned)((per_g + 255) / 256), c.G);
    if (c.B > 1)
        landmark_unpermute_kernel<float4, 4><<<grid, 256, 0, s>>>((const float4*)c.lm[layer], (float4*)dst, c.Cmax,
                                                                  c.d / 4);
    else
        landmark_unpermute_kernel<uint4, 8><<<grid, 256, 0, s>>>((const uint4*)c.lm[layer], (uint4*)dst, c.Cmax,
                                                                 c.d / 8);
    return cudaGetLastError();
}

// ------------------------------------------------------------- selection
// Thread t of a 256-thread CTA owns radix bin 255 - t (descending).  Given
// per-bin counts, find the bin holding the k_rem-th largest key: its digit,
// the keys still wanted from it and its count (when the two are equal the
// whole bin is taken and the search can end).
__device__ __forceinline__ void pick_digit_cnt(uint32_t cnt, uint32_t* warp_sums, int* s_digit, uint32_t* s_krem,
                                               uint32_t* s_bincnt, uint32_t k_rem) {
    uint32_t total;
    const uint32_t excl = block_exclusive_scan(cnt, warp_sums, &total);
    if (excl < k_rem && excl + cnt >= k_rem) {
        *s_digit = 255 - (int)threadIdx.x;
        *s_krem = k_rem - excl;
        *s_bincnt = cnt;
    }
    __syncthreads();
}

// resident CTAs per SM requested (a register budget): measured on the four
// large workloads, 4 for fp32 landmarks and none for bf16 ones, whose deeper
// per-thread load batches beat occupancy
template <bool BF16LM, int SEL_RPT>
constexpr int sel_min_blocks() { return SEL_RPT == 1 ? 4 : (BF16LM ? (SEL_RPT == 2 ? 2 : 1) : 4); }

// The group's summed query (and speculative query with DUAL), fp32, into u_s.
template <int D, bool DUAL>
__device__ __forceinline__ void sum_queries(const uint16_t* __restrict__ q, const uint16_t* __restrict__ qs, int b,
                                            int g, int Hq, int r, float (*u_s)[D]) {
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        const uint16_t* qp = q + ((int64_t)b * Hq + g * r) * D + c;
        float a = 0.f;
        for (int h = 0; h < r; ++h) a += __uint_as_float((uint32_t)qp[h * D] << 16);
        u_s[0][c] = a;
        if (DUAL) {
            const uint16_t* sp = qs + ((int64_t)b * Hq + g * r) * D + c;
            float e = 0.f;
            for (int h = 0; h < r; ++h) e += __uint_as_float((uint32_t)sp[h * D] << 16);
            u_s[1][c] = e;
        }
    }
}

// Bulk L2 prefetch of the first pf_chunks 16-byte chunks of landmark rows
// [row0, row0 + nrows) of group bg (one contiguous run of 16 * nrows bytes per
// chunk), issued by the first warp before the CTA sums its query, so the
// landmark bytes stream from HBM while that prologue runs.
template <int D, bool BF16LM>
__device__ __forceinline__ void prefetch_rows_l2(const void* lm_v, int bg, int Cmax, int row0, int nrows,
                                                 int pf_chunks) {
    constexpr int NCH = BF16LM ? D / 8 : D / 4;
    if (threadIdx.x >= 32 || nrows <= 0) return;
    const char* g0 = reinterpret_cast<const char*>(lm_v) + ((int64_t)bg * NCH * Cmax + row0) * 16;
    for (int c = threadIdx.x; c < min(pf_chunks, NCH); c += 32)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(g0 + (int64_t)c * Cmax * 16),
                     "r"((uint32_t)nrows * 16u)
                     : "memory");
}

// Scores of SEL_RPT landmark rows per thread (rows row0 + i * SEL_THREADS,
// those at or past C scoring 0) against the NQ summed queries in u_s.
template <int D, bool BF16LM, int NQ, int SEL_RPT>
__device__ __forceinline__ void score_rows(const void* __restrict__ lm_v, int bg, int Cmax, int C, int row0,
                                           const float (*u_s)[D], float (&acc)[NQ][SEL_RPT]) {
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int i = 0; i < SEL_RPT; ++i) acc[qi][i] = 0.f;

    if (!BF16LM) {
        const float4* lm = reinterpret_cast<const float4*>(lm_v) + (int64_t)bg * (D / 4) * Cmax;
#pragma unroll 4
        for (int c4 = 0; c4 < D / 4; ++c4) {
            float4 v[SEL_RPT];
#pragma unroll
            for (int i = 0; i < SEL_RPT; ++i) {
                const int j = row0 + i * SEL_THREADS;
                v[i] = j < C ? __ldg(lm + (int64_t)c4 * Cmax + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const float4 u = *reinterpret_cast<const float4*>(&u_s[qi][4 * c4]);
#pragma unroll
                for (int i = 0; i < SEL_RPT; ++i) {
                    float a = acc[qi][i];
                    a = fmaf(v[i].x, u.x, a);
                    a = fmaf(v[i].y, u.y, a);
                    a = fmaf(v[i].z, u.z, a);
                    a = fmaf(v[i].w, u.w, a);
                    acc[qi][i] = a;
                }
            }
        }
    } else {
        const uint4* lm = reinterpret_cast<const uint4*>(lm_v) + (int64_t)bg * (D / 8) * Cmax;
#pragma unroll 4
        for (int c8 = 0; c8 < D / 8; ++c8) {
            uint4 v[SEL_RPT];
#pragma unroll
            for (int i = 0; i < SEL_RPT; ++i) {
                const int j = row0 + i * SEL_THREADS;
                v[i] = j < C ? __ldg(lm + (int64_t)c8 * Cmax + j) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const float4 u0 = *reinterpret_cast<const float4*>(&u_s[qi][8 * c8]);
                const float4 u1 = *reinterpret_cast<const float4*>(&u_s[qi][8 * c8 + 4]);
#pragma unroll
                for (int i = 0; i < SEL_RPT; ++i) {
                    float a = acc[qi][i];
                    a = fmaf(bf16lo_to_f32(v[i].x), u0.x, a);
                    a = fmaf(bf16hi_to_f32(v[i].x), u0.y, a);
                    a = fmaf(bf16lo_to_f32(v[i].y), u0.z, a);
                    a = fmaf(bf16hi_to_f32(v[i].y), u0.w, a);
                    a = fmaf(bf16lo_to_f32(v[i].z), u1.x, a);
                    a = fmaf(bf16hi_to_f32(v[i].z), u1.y, a);
                    a = fmaf(bf16lo_to_f32(v[i].w), u1.z, a);
                    a = fmaf(bf16hi_to_f32(v[i].w), u1.w, a);
                    acc[qi][i] = a;
                }
            }
        }
    }
}

// ASSIGN: the last CTA of a group then assigns the group's resident slots for
// its true index (the routine of resident_assign.cuh, `aa` with need = the
// true index; res_assign_ints(k) ints of dynamic shared memory), so a step
// without a speculative query needs no separate assignment launch.
template <int D, bool BF16LM, bool DUAL, int SEL_RPT, bool ASSIGN>
__global__ void __launch_bounds__(SEL_THREADS, sel_min_blocks<BF16LM, SEL_RPT>())
select_kernel(const void* __restrict__ lm_v, const uint16_t* __restrict__ q, const uint16_t* __restrict__ qs,
              const int2* __restrict__ items, const int32_t* __restrict__ nchunks, const int32_t* __restrict__ g_C,
              uint32_t* __restrict__ keys, uint32_t* __restrict__ hist, uint32_t* __restrict__ done,
              int32_t* __restrict__ idx_true, int32_t* __restrict__ idx_pred, int G, int Cmax4, int Cmax, int r,
              int Hkv, int k, int key_cache, int dep_wait, int pf_chunks, const ResAssignArgs aa) {
    constexpr int NQ = DUAL ? 2 : 1;
    __shared__ __align__(16) float u_s[NQ][D];
    __shared__ uint32_t h_s[NQ][256];
    __shared__ uint32_t warp_sums[32];
    __shared__ int s_last;
    __shared__ int s_digit;
    __shared__ uint32_t s_krem, s_bincnt;

    const int tid = threadIdx.x;
    // dep_wait: launched as a programmatic dependent of the kernel before it on
    // the stream, which may have written any input (and a selection before it
    // resets the histograms and tickets last) -- nothing is read before it is done
    if (dep_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int2 it = items[blockIdx.x];
    const int bg = it.x, chunk = it.y;
    const int b = bg / Hkv, g = bg % Hkv;
    const int C = g_C[bg];
    const int Hq = Hkv * r;
    prefetch_rows_l2<D, BF16LM>(lm_v, bg, Cmax, chunk * SEL_THREADS * SEL_RPT,
                                min(SEL_THREADS * SEL_RPT, C - chunk * SEL_THREADS * SEL_RPT), pf_chunks);

    sum_queries<D, DUAL>(q, qs, b, g, Hq, r, u_s);
    for (int i = tid; i < NQ * 256; i += SEL_THREADS) (&h_s[0][0])[i] = 0u;
    __syncthreads();

    // ---- score SEL_RPT rows per thread (rows strided by the CTA width)
    constexpr int SEL_ROWS = SEL_THREADS * SEL_RPT;
    const int row0 = chunk * SEL_ROWS + tid;
    float acc[NQ][SEL_RPT];
    score_rows<D, BF16LM, NQ, SEL_RPT>(lm_v, bg, Cmax, C, row0, u_s, acc);
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        uint32_t* kq = keys + ((int64_t)qi * G + bg) * Cmax4;
#pragma unroll
        for (int i = 0; i < SEL_RPT; ++i) {
            const int j = row0 + i * SEL_THREADS;
            if (j < C) {
                const uint32_t key = float_to_ordered(acc[qi][i]);
                kq[j] = key;
                atomicAdd(&h_s[qi][key >> 24], 1u);
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < NQ * 256; i += SEL_THREADS) {
        const uint32_t v = (&h_s[0][0])[i];
        if (v) atomicAdd(&hist[((int64_t)(i / 256) * G + bg) * 256 + (i % 256)], v);
    }
    // the kernel behind this one may be scheduled once every CTA has scored
    if (dep_wait) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the CTA's key and histogram writes reach thread 0 through the barrier; its
    // release fence orders them before the ticket, the last CTA's acquire fence
    // orders the selection's loads after it
    __syncthreads();
    if (tid == 0) {
        fence_acq_rel_gpu();
        const uint32_t prev = atomicAdd(&done[bg], 1u);
        s_last = (prev + 1 == (uint32_t)nchunks[bg]);
        if (s_last) fence_acq_rel_gpu();
    }
    __syncthreads();
    if (!s_last) return;

    // ---- last CTA of the group: exact top-k for each query.  Thread t owns the
    // contiguous keys [c0, c1) of the group (a multiple of 4 of them, so 16-byte
    // loads stay inside the padded key row), read 16 at a time with independent
    // loads; the compaction then needs two block scans in all.  With key_cache
    // the group's keys are first copied into shared memory (one round trip to
    // L2), and the radix passes and the compaction read them there.
    extern __shared__ __align__(16) uint32_t sel_dyn[];
    const int per = ((C + SEL_THREADS - 1) / SEL_THREADS + 3) & ~3;
    const int c0 = min(C, tid * per), c1 = min(C, c0 + per);
    for (int qi = 0; qi < NQ; ++qi) {
        const uint32_t* kq = keys + ((int64_t)qi * G + bg) * Cmax4;
        if (key_cache) {
            for (int i = 4 * tid; i < C; i += 4 * SEL_THREADS)
                *reinterpret_cast<uint4*>(sel_dyn + i) = __ldcg(reinterpret_cast<const uint4*>(kq + i));
            __syncthreads();
            kq = sel_dyn;
        }
        int32_t* out = (qi == 0 ? idx_true : idx_pred) + (int64_t)bg * k;
        uint32_t* hg = hist + ((int64_t)qi * G + bg) * 256;
        uint32_t k_rem = (uint32_t)min(k, C);
        const uint32_t cnt0 = __ldcg(hg + 255 - tid);
        hg[255 - tid] = 0u;                                  // leave the histogram zeroed
        pick_digit_cnt(cnt0, warp_sums, &s_digit, &s_krem, &s_bincnt, k_rem);
        uint32_t prefix = (uint32_t)s_digit << 24, mask = 0xFF000000u;
        bool whole_bin = s_krem == s_bincnt;                  // the bin's keys are all wanted: done
        k_rem = s_krem;
        // four keys from the cache or from L2
        auto ld4 = [&](int j) -> uint4 {
            return key_cache ? *reinterpret_cast<const uint4*>(kq + j) : __ldcg(reinterpret_cast<const uint4*>(kq + j));
        };
        // visit this thread's keys in ascending order: f(j, key)
        auto scan_chunk = [&](auto&& f) {
            for (int j = c0; j < c1; j += 16) {
                uint4 kv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) kv[u] = j + 4 * u < c1 ? ld4(j + 4 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t kk[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (j + 4 * u + e < c1) f(j + 4 * u + e, kk[e]);
                }
            }
        };
        const bool small = C <= 4 * SEL_THREADS;             // at most 4 keys per thread
        for (int shift = 16; shift >= 0 && !whole_bin; shift -= 8) {
            h_s[0][tid] = 0u;
            __syncthreads();
            if (small) {
                const int j0 = 4 * tid;
                if (j0 < C) {
                    const uint4 kv4 = ld4(j0);
                    const uint32_t kv[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (j0 + e < C && (kv[e] & mask) == prefix) atomicAdd(&h_s[0][(kv[e] >> shift) & 0xFFu], 1u);
                }
            } else {
                scan_chunk([&](int, uint32_t key) {
                    if ((key & mask) == prefix) atomicAdd(&h_s[0][(key >> shift) & 0xFFu], 1u);
                });
            }
            __syncthreads();
            const uint32_t cnt = h_s[0][255 - tid];
            __syncthreads();
            pick_digit_cnt(cnt, warp_sums, &s_digit, &s_krem, &s_bincnt, k_rem);
            prefix |= (uint32_t)s_digit << shift;
            mask |= 0xFFu << shift;
            whole_bin = s_krem == s_bincnt;
            k_rem = s_krem;
        }
        // under the mask, prefix is the k-th largest key: take every key above it
        // and the first k_rem equal to it (all of them when the search ended on a
        // whole bin), in ascending id order
        const uint32_t thr = prefix;
        const uint32_t k_eq = k_rem;
        if (small) {
            // one sweep: 4 keys per thread in id order, two block scans
            const int j0 = 4 * tid;
            uint4 kv4 = make_uint4(0u, 0u, 0u, 0u);
            if (j0 < C) kv4 = ld4(j0);
            const uint32_t kv[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
            uint32_t n_eq = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) n_eq += (j0 + e < C && (kv[e] & mask) == thr);
            uint32_t tot;
            uint32_t eq_run = block_exclusive_scan(n_eq, warp_sums, &tot);
            uint32_t sel = 0;
            bool take[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool valid = j0 + e < C;
                bool t = valid && (kv[e] & mask) > thr;
                if (valid && (kv[e] & mask) == thr) t = eq_run++ < k_eq;
                take[e] = t;
                sel += t;
            }
            uint32_t pos = block_exclusive_scan(sel, warp_sums, &tot);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (take[e]) out[pos++] = j0 + e;
        } else {
            // counts per chunk, two block scans for the offsets, then the writes
            uint32_t n_gt = 0, n_eq = 0;
            scan_chunk([&](int, uint32_t key) {
                n_gt += (key & mask) > thr;
                n_eq += (key & mask) == thr;
            });
            uint32_t tot;
            const uint32_t eq_before = block_exclusive_scan(n_eq, warp_sums, &tot);
            const uint32_t eq_take = eq_before >= k_eq ? 0u : min(n_eq, k_eq - eq_before);
            uint32_t pos = block_exclusive_scan(n_gt + eq_take, warp_sums, &tot);
            uint32_t eq_run = eq_before;
            scan_chunk([&](int j, uint32_t key) {
                bool take = (key & mask) > thr;
                if ((key & mask) == thr) take = eq_run++ < k_eq;
                if (take) out[pos++] = j;
            });
        }
        __syncthreads();
    }
    if (tid == 0) done[bg] = 0u;
    if constexpr (ASSIGN) {
        // the true index this CTA wrote is visible to all its threads after the
        // barrier that closed the loop above
        extern __shared__ __align__(16) int32_t sel_rs[];
        __shared__ uint32_t s_tot;
        resident_assign_group(aa, bg, sel_rs, warp_sums, &s_tot);
    }
}

// Cluster selection: a group's landmark rows are split over the S CTAs of one
// thread-block cluster (S <= 8; rank r scores rows [r * SEL_ROWS, (r + 1) *
// SEL_ROWS)), each CTA keeping its keys in its own shared memory.  The radix
// select runs on all S CTAs at once: every pass each CTA histograms the digit
// of its own keys that still match the prefix, a cluster barrier publishes the
// histograms, and every CTA sums the S histograms of a bin through distributed
// shared memory and picks the same digit.  A pass whose bin holds exactly the
// keys still wanted ends the search early (they are all taken).  The winners
// are written in ascending id order: each CTA publishes its counts of keys
// above and equal to the threshold, and offsets its writes by those of the
// lower ranks.  No keys, histograms or tickets go through global memory.
// With ASSIGN, rank 0 assigns the group's resident slots once every rank's
// writes of the true index are visible to it (the release / acquire cluster
// barrier).
template <int D, bool BF16LM, bool DUAL, int SEL_RPT, bool ASSIGN>
__global__ void __launch_bounds__(SEL_THREADS, sel_min_blocks<BF16LM, SEL_RPT>())
select_cluster_kernel(const void* __restrict__ lm_v, const uint16_t* __restrict__ q, const uint16_t* __restrict__ qs,
                      const int32_t* __restrict__ g_C, int32_t* __restrict__ idx_true, int32_t* __restrict__ idx_pred,
                      int Cmax, int r, int Hkv, int k, int dep_wait, int pf_chunks, const ResAssignArgs aa) {
    constexpr int NQ = DUAL ? 2 : 1;
    constexpr int SEL_ROWS = SEL_THREADS * SEL_RPT;
    __shared__ __align__(16) float u_s[NQ][D];
    __shared__ __align__(16) uint32_t k_s[NQ][SEL_ROWS];   // this CTA's keys, local row order
    __shared__ uint32_t h_s[NQ][256];                        // top-byte histogram of this CTA's keys
    __shared__ uint32_t hc[2][256];                          // later passes' histograms, alternating
    __shared__ uint32_t cnt_s[NQ][2];                        // keys above / equal to the threshold
    __shared__ uint32_t warp_sums[32];
    __shared__ int s_digit;
    __shared__ uint32_t s_krem, s_bincnt;

    const int tid = threadIdx.x;
    if (dep_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t S = cluster_size(), rank = cluster_rank();
    const int bg = (int)(blockIdx.x / S);
    const int b = bg / Hkv, g = bg % Hkv;
    const int C = g_C[bg];
    const int base = (int)rank * SEL_ROWS;                   // first row of this CTA
    const int nloc = max(0, min(C - base, SEL_ROWS));        // rows of this CTA
    prefetch_rows_l2<D, BF16LM>(lm_v, bg, Cmax, base, nloc, pf_chunks);

    sum_queries<D, DUAL>(q, qs, b, g, Hkv * r, r, u_s);
    for (int i = tid; i < NQ * 256; i += SEL_THREADS) (&h_s[0][0])[i] = 0u;
    __syncthreads();

    float acc[NQ][SEL_RPT];
    score_rows<D, BF16LM, NQ, SEL_RPT>(lm_v, bg, Cmax, C, base + tid, u_s, acc);
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int i = 0; i < SEL_RPT; ++i) {
            const int j = tid + i * SEL_THREADS;
            if (j < nloc) {
                const uint32_t key = float_to_ordered(acc[qi][i]);
                k_s[qi][j] = key;
                atomicAdd(&h_s[qi][key >> 24], 1u);
            }
        }
    // the kernel behind this one may be scheduled once every CTA has scored
    if (dep_wait) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    cluster_barrier();                                       // keys and top-byte histograms complete

    // thread t's keys for the passes and the compaction: local rows
    // [t * SEL_RPT, (t + 1) * SEL_RPT), in id order
    const int j0 = tid * SEL_RPT;
    for (int qi = 0; qi < NQ; ++qi) {
        uint32_t kr[SEL_RPT];
        if constexpr (SEL_RPT == 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(&k_s[qi][j0]);
            kr[0] = v.x; kr[1] = v.y; kr[2] = v.z; kr[3] = v.w;
        } else if constexpr (SEL_RPT == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(&k_s[qi][j0]);
            kr[0] = v.x; kr[1] = v.y;
        } else {
            kr[0] = k_s[qi][j0];
        }
        const int n_mine = min(SEL_RPT, max(0, nloc - j0));
        int32_t* out = (qi == 0 ? idx_true : idx_pred) + (int64_t)bg * k;
        uint32_t k_rem = (uint32_t)min(k, C);
        if (k_rem == 0) continue;                            // the same for every rank of the cluster
        uint32_t prefix = 0u, mask = 0u;
        const uint32_t* hsrc = h_s[qi];
        int shift = 24, hb = 0;
        while (true) {
            uint32_t cnt = 0;
            for (uint32_t rr = 0; rr < S; ++rr) cnt += ld_cluster_u32(hsrc + 255 - tid, rr);
            // the buffer the next pass fills: its last remote readers passed the barrier before this pass
            hc[hb][tid] = 0u;
            pick_digit_cnt(cnt, warp_sums, &s_digit, &s_krem, &s_bincnt, k_rem);
            prefix |= (uint32_t)s_digit << shift;
            mask |= 0xFFu << shift;
            const bool whole_bin = s_krem == s_bincnt;
            k_rem = s_krem;
            if (shift == 0 || whole_bin) break;              // the same decision on every rank
            shift -= 8;
#pragma unroll
            for (int e = 0; e < SEL_RPT; ++e)
                if (e < n_mine && (kr[e] & mask) == prefix) atomicAdd(&hc[hb][(kr[e] >> shift) & 0xFFu], 1u);
            cluster_barrier();
            hsrc = hc[hb];
            hb ^= 1;
        }
        // take every key whose masked value is above the prefix and the first
        // k_rem equal to it (all of them when the search ended on a whole bin)
        const uint32_t k_eq = k_rem;
        uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
        for (int e = 0; e < SEL_RPT; ++e)
            if (e < n_mine) {
                n_gt += (kr[e] & mask) > prefix;
                n_eq += (kr[e] & mask) == prefix;
            }
        uint32_t tot_eq, tot_gt;
        const uint32_t eq_excl = block_exclusive_scan(n_eq, warp_sums, &tot_eq);
        const uint32_t gt_excl = block_exclusive_scan(n_gt, warp_sums, &tot_gt);
        if (tid == 0) {
            cnt_s[qi][0] = tot_gt;
            cnt_s[qi][1] = tot_eq;
        }
        cluster_barrier();                                   // every rank's counts published
        uint32_t pos_base = 0, eq_base = 0;
        for (uint32_t rr = 0; rr < rank; ++rr) {
            const uint32_t gt_r = ld_cluster_u32(&cnt_s[qi][0], rr), eq_r = ld_cluster_u32(&cnt_s[qi][1], rr);
            pos_base += gt_r + (eq_base >= k_eq ? 0u : min(eq_r, k_eq - eq_base));
            eq_base += eq_r;
        }
        // thread t writes after the lower ranks' winners, this CTA's keys above
        // the threshold before it and its equal keys taken before it
        uint32_t eq_run = eq_base + eq_excl;
        uint32_t pos = pos_base + gt_excl + (eq_base >= k_eq ? 0u : min(eq_excl, k_eq - eq_base));
#pragma unroll
        for (int e = 0; e < SEL_RPT; ++e)
            if (e < n_mine) {
                const uint32_t m = kr[e] & mask;
                bool take = m > prefix;
                if (m == prefix) take = eq_run++ < k_eq;
                if (take) out[pos++] = base + j0 + e;
            }
    }
    // no CTA leaves while another may still read its shared memory; with
    // ASSIGN the barrier also makes every rank's index writes visible to rank 0
    cluster_barrier();
    if constexpr (ASSIGN) {
        if (rank == 0) {
            extern __shared__ __align__(16) int32_t sel_rs[];
            __shared__ uint32_t s_tot;
            resident_assign_group(aa, bg, sel_rs, warp_sums, &s_tot);
        }
    }
}

cudaError_t launch_select(const Ctx& c, int layer, const void* q, const void* q_spec, int32_t* idx_true,
                          int32_t* idx_pred, cudaStream_t s, const ResAssignArgs* assign, bool pdl) {
    const int Cmax4 = (c.Cmax + 3) & ~3;
    const bool dual = q_spec != nullptr;
    const bool bf = c.B == 1;
    if (assign && dual) return cudaErrorInvalidValue;     // the fused assignment is for single-query steps
    ResAssignArgs aa{};
    size_t dyn = 0;
    if (assign) {
        aa = *assign;
        aa.need = idx_true;
        dyn = sizeof(int32_t) * res_assign_ints(c.k);
    }
    // the last CTA's key cache (the same shared memory the assignment uses after it)
    const int key_cache = Cmax4 <= SEL_KEY_CACHE ? 1 : 0;
    if (key_cache) dyn = std::max(dyn, sizeof(uint32_t) * (size_t)Cmax4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c.n_sel_items);
    cfg.blockDim = dim3(SEL_THREADS);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int dep_wait = pdl ? 1 : 0;
    // Grids of more than one wave prefetch the first chunks of each CTA's rows
    // into the L2 up front (as many as keep the resident CTAs' prefetched
    // bytes within 48 MB of the 129 MB L2): a CTA of a later wave then streams
    // while it sums its query.  Long-context layer (2.5 waves): 135.3 ->
    // 129.7 us.  One-wave grids start every CTA at once and gained nothing
    // (Llama layer 16.4-16.5 -> 16.7 us, wide budget 39.7-39.9 -> 40.2 us).
    const int64_t rows_cta = (int64_t)SEL_THREADS * c.sel_rpt;
    const int64_t grid_ctas = c.sel_clu > 0 ? (int64_t)c.G * c.sel_clu : c.n_sel_items;
    const int64_t resident = std::min<int64_t>(grid_ctas, 4 * (int64_t)c.sel_sms);
    const int pf_chunks = grid_ctas <= resident ? 0 :
        (int)std::min<int64_t>(bf ? c.d / 8 : c.d / 4, (48ll << 20) / std::max<int64_t>(1, resident * rows_cta * 16));
    cudaError_t err = cudaSuccess;
    if (c.sel_clu > 0) {
        // one cluster of sel_clu CTAs per group; only the assignment's lists are dynamic
        cudaLaunchAttribute ca[2];
        ca[0].id = cudaLaunchAttributeClusterDimension;
        ca[0].val.clusterDim.x = (unsigned)c.sel_clu;
        ca[0].val.clusterDim.y = 1;
        ca[0].val.clusterDim.z = 1;
        ca[1] = attr[0];
        cfg.gridDim = dim3((unsigned)(c.G * c.sel_clu));
        cfg.dynamicSmemBytes = assign ? sizeof(int32_t) * res_assign_ints(c.k) : 0;
        cfg.attrs = ca;
        cfg.numAttrs = pdl ? 2 : 1;
#define KVO_SELC_L(D_, BF_, DU_, RPT_, AS_)                                                                    \
    err = cudaLaunchKernelEx(&cfg, select_cluster_kernel<D_, BF_, DU_, RPT_, AS_>, c.lm[layer],                \
                             (const uint16_t*)q, (const uint16_t*)q_spec, (const int32_t*)c.g_C, idx_true,     \
                             idx_pred, c.Cmax, c.r, c.Hkv, c.k, dep_wait, pf_chunks, aa)
#define KVO_SELC(D_, BF_, DU_, AS_)                                                                            \
    do {                                                                                                       \
        if (c.sel_rpt == 1) KVO_SELC_L(D_, BF_, DU_, 1, AS_);                                                  \
        else if (c.sel_rpt == 2) KVO_SELC_L(D_, BF_, DU_, 2, AS_);                                             \
        else KVO_SELC_L(D_, BF_, DU_, 4, AS_);                                                                 \
    } while (0)
        if (assign) {
            if (c.d == 128) { if (bf) KVO_SELC(128, true, false, true); else KVO_SELC(128, false, false, true); }
            else            { if (bf) KVO_SELC(64, true, false, true); else KVO_SELC(64, false, false, true); }
        } else if (c.d == 128) {
            if (bf) { if (dual) KVO_SELC(128, true, true, false); else KVO_SELC(128, true, false, false); }
            else    { if (dual) KVO_SELC(128, false, true, false); else KVO_SELC(128, false, false, false); }
        } else {
            if (bf) { if (dual) KVO_SELC(64, true, true, false); else KVO_SELC(64, true, false, false); }
            else    { if (dual) KVO_SELC(64, false, true, false); else KVO_SELC(64, false, false, false); }
        }
#undef KVO_SELC
#undef KVO_SELC_L
        return err;
    }
#define KVO_SEL_L(D_, BF_, DU_, RPT_, AS_)                                                                     \
    err = cudaLaunchKernelEx(&cfg, select_kernel<D_, BF_, DU_, RPT_, AS_>, c.lm[layer], (const uint16_t*)q,     \
                             (const uint16_t*)q_spec, (const int2*)c.sel_items, (const int32_t*)c.sel_nchunks,  \
                             (const int32_t*)c.g_C, c.sel_keys, c.sel_hist, c.sel_done, idx_true, idx_pred, c.G, \
                             Cmax4, c.Cmax, c.r, c.Hkv, c.k, key_cache, dep_wait, pf_chunks, aa)
#define KVO_SEL(D_, BF_, DU_)                                                                                  \
    do {                                                                                                       \
        if (c.sel_rpt == 1) KVO_SEL_L(D_, BF_, DU_, 1, false);                                                  \
        else if (c.sel_rpt == 2) KVO_SEL_L(D_, BF_, DU_, 2, false);                                             \
        else KVO_SEL_L(D_, BF_, DU_, 4, false);                                                                \
    } while (0)
#define KVO_SEL_A(D_, BF_)                                                                                     \
    do {                                                                                                       \
        if (c.sel_rpt == 1) KVO_SEL_L(D_, BF_, false, 1, true);                                                \
        else if (c.sel_rpt == 2) KVO_SEL_L(D_, BF_, false, 2, true);                                           \
        else KVO_SEL_L(D_, BF_, false, 4, true);                                                               \
    } while (0)
    if (assign) {
        if (c.d == 128) { if (bf) KVO_SEL_A(128, true); else KVO_SEL_A(128, false); }
        else            { if (bf) KVO_SEL_A(64, true); else KVO_SEL_A(64, false); }
    } else if (c.d == 128) {
        if (bf) { if (dual) KVO_SEL(128, true, true); else KVO_SEL(128, true, false); }
        else    { if (dual) KVO_SEL(128, false, true); else KVO_SEL(128, false, false); }
    } else {
        if (bf) { if (dual) KVO_SEL(64, true, true); else KVO_SEL(64, true, false); }
        else    { if (dual) KVO_SEL(64, false, true); else KVO_SEL(64, false, false); }
    }
#undef KVO_SEL_A
#undef KVO_SEL
#undef KVO_SEL_L
    return err;
}

// Dynamic shared memory of the fused selection + assignment kernels (the
// assignment's lists or the key cache, whichever is larger; above the default
// 48 KB only for k > 2457).
cudaError_t prepare_select_assign(const Ctx& c) {
    const int Cmax4 = (c.Cmax + 3) & ~3;
    const int bytes = (int)std::max(sizeof(int32_t) * res_assign_ints(c.k),
                                    Cmax4 <= SEL_KEY_CACHE ? sizeof(uint32_t) * (size_t)Cmax4 : (size_t)0);
    cudaError_t e = cudaSuccess;
#define KVO_SEL_ATTR(D_, BF_, RPT_)                                                                            \
    if (e == cudaSuccess)                                                                                      \
        e = cudaFuncSetAttribute(select_kernel<D_, BF_, false, RPT_, true>,                                    \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)
    KVO_SEL_ATTR(128, true, 1); KVO_SEL_ATTR(128, true, 2); KVO_SEL_ATTR(128, true, 4);
    KVO_SEL_ATTR(128, false, 1); KVO_SEL_ATTR(128, false, 2); KVO_SEL_ATTR(128, false, 4);
    KVO_SEL_ATTR(64, true, 1); KVO_SEL_ATTR(64, true, 2); KVO_SEL_ATTR(64, true, 4);
    KVO_SEL_ATTR(64, false, 1); KVO_SEL_ATTR(64, false, 2); KVO_SEL_ATTR(64, false, 4);
#undef KVO_SEL_ATTR
    const int abytes = (int)(sizeof(int32_t) * res_assign_ints(c.k));
#define KVO_SELC_ATTR(D_, BF_, RPT_)                                                                           \
    if (e == cudaSuccess)                                                                                      \
        e = cudaFuncSetAttribute(select_cluster_kernel<D_, BF_, false, RPT_, true>,                            \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, abytes)
    KVO_SELC_ATTR(128, true, 1); KVO_SELC_ATTR(128, true, 2); KVO_SELC_ATTR(128, true, 4);
    KVO_SELC_ATTR(128, false, 1); KVO_SELC_ATTR(128, false, 2); KVO_SELC_ATTR(128, false, 4);
    KVO_SELC_ATTR(64, true, 1); KVO_SELC_ATTR(64, true, 2); KVO_SELC_ATTR(64, true, 4);
    KVO_SELC_ATTR(64, false, 1); KVO_SELC_ATTR(64, false, 2); KVO_SELC_ATTR(64, false, 4);
#undef KVO_SELC_ATTR
    return e;
}

}  // namespace kvo
