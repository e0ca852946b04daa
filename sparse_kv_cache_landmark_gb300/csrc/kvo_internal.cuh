// Internal declarations shared by the CUDA translation units of libkvo.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "kvo.h"

namespace kvo {

// ---------------------------------------------------------------- tunables
constexpr int SEL_THREADS = 256;          // select: threads per CTA
constexpr int SEL_KEY_CACHE = 8192;       // select: keys per group the last CTA stages in shared memory (32 KB)
constexpr int SEL_RPT_MAX = 4;            // select: landmark rows per thread (1 or 4, chosen at init)
constexpr int ATT_WARPS = 4;              // attention: warps per CTA
constexpr int ATT_TILE = 16;              // attention: tokens per mma tile
constexpr int ATT_TILES_PER_ITEM = 16;    // attention: tiles per CTA work item
constexpr int GATHER_THREADS = 256;
constexpr int TMA_STAGE_BYTES = 16384;    // TMA gather: bytes per batch
constexpr int TMA_MAX_PIECES = 64;        // TMA gather: pieces per batch
__host__ __device__ constexpr size_t tma_driver_smem(int stages) {
    return (size_t)stages * TMA_STAGE_BYTES + (size_t)stages * TMA_MAX_PIECES * 24 + (size_t)stages * 12 + 16;
}

// ------------------------------------------------------------------ context
struct Ctx {
    kvo_config cfg{};
    std::vector<int32_t> lens;
    int G = 0, r = 0, d = 0, B = 0, k = 0, W = 0, L = 0, Hkv = 0, Hq = 0, batch = 0;
    int Cmax = 0;
    // per group (device): element offset of the group's rows in the packed host
    // arrays, candidate blocks C_b, context length len_b
    int64_t* g_off = nullptr;
    int32_t* g_C = nullptr;
    std::vector<const uint16_t*> k_host, v_host;   // device-addressable host pointers
    std::vector<const uint16_t*> k_win, v_win;     // window per layer ([G][Wcap][d]; the ring in append mode)
    int Wcap = 0;                   // window storage per group: W, or W + B in append mode
    int max_append = 0, appended = 0;
    int32_t* g_len = nullptr;       // [G] current context length (append mode)
    int32_t* g_wstart = nullptr;    // [G] ring slot of the window's first token (append mode)
    int32_t* g_wlen = nullptr;      // [G] window length (append mode)
    std::vector<uint16_t*> ring_k, ring_v;   // library-owned window rings (append mode)
    uint16_t** d_ring_k = nullptr;  // device copies of the per-layer pointer tables
    uint16_t** d_ring_v = nullptr;
    uint16_t** d_host_k = nullptr;
    uint16_t** d_host_v = nullptr;
    void** d_lm = nullptr;
    std::vector<void*> lm;                          // landmarks per layer
    size_t lm_bytes = 0;
    uint16_t* pp_k[2] = {nullptr, nullptr};
    uint16_t* pp_v[2] = {nullptr, nullptr};
    size_t pp_bytes = 0;
    // Resident mode (cross-step delta prefetch): one persistent block set of 2k
    // slots per layer and group, laid out like a ping-pong half.
    bool resident = false;
    std::vector<uint16_t*> res_k, res_v;   // [L] -> [G][2k][B][d]
    int32_t* res_map = nullptr;     // [L][G][Ccap] slot of each block, -1 when not resident
    int32_t* res_slots = nullptr;   // [L][G][2k] block held by each slot, -1 when empty
    int32_t* res_dslot = nullptr;   // [L][G][k] urgent fetches: destination slots
    int32_t* res_pf_ids = nullptr;  // [L][G][k] prefetch fetches: block ids
    int32_t* res_pf_cnt = nullptr;  // [L][G]
    int32_t* res_pf_dslot = nullptr;// [L][G][k]
    unsigned long long* res_fetched = nullptr;   // [2] blocks fetched: urgent, prefetch
    std::vector<char> res_pending;  // [L] a prefetch into the layer's set was issued and not yet waited for
    int res_budget = -1;            // prefetch fetches admitted per group, layer and step (-1: all)
    // speculation policy: 0 prefetch every layer's prediction; 1 per layer, only
    // while its prefetches pay (kvo_set_spec_policy)
    int spec_policy = 0;
    uint8_t* res_pfbit = nullptr;             // [L][G][2k] slot filled by a prefetch, not used yet
    unsigned long long* res_stat = nullptr;   // [L][2] blocks prefetched, prefetched blocks used (since init)
    unsigned long long* res_pol = nullptr;    // [L][8] policy state: on, steps, window fetched, window used, rest
    uint32_t* res_pol_ticket = nullptr;       // [L] last-CTA tickets of the policy update (zero between launches)
    // chain steps: attention over the blocks resident already (and the window)
    // beside the urgent copies, then over the fetched ones, merged by lse
    int32_t* res_hit_slot = nullptr;  // [G][k] slots of the hits, in index order
    int32_t* res_hit_cnt = nullptr;   // [G]
    float* res_oA = nullptr;          // [rows][d], [rows]: hits + window
    float* res_lA = nullptr;
    // partials of the fetched-block attention when a group spans several CTAs
    float* mp_part_o = nullptr;       // [G][S][r][d]
    float* mp_part_ml = nullptr;      // [G][S][r][2]
    uint32_t* mp_done = nullptr;      // [G] tickets (zero between launches)
    // Low-rank keys per layer (caller-owned device factors; rank 0: not set)
    std::vector<const uint16_t*> lr_coef, lr_basis;
    std::vector<int> lr_rank;
    // K / V buffer by id: 0, 1 ping-pong halves; 2 + l resident set of layer l
    uint16_t* buf_k(int buf) const { return buf < 2 ? pp_k[buf] : res_k[buf - 2]; }
    uint16_t* buf_v(int buf) const { return buf < 2 ? pp_v[buf] : res_v[buf - 2]; }
    // select scratch
    uint32_t* sel_keys = nullptr;   // [2][G][Cmax]
    uint32_t* sel_hist = nullptr;   // [2][G][256]
    uint32_t* sel_done = nullptr;   // [G]
    int2* sel_items = nullptr;      // {group, chunk}
    int32_t* sel_nchunks = nullptr; // [G]
    int n_sel_items = 0;
    int sel_rpt = 4;                // rows per thread of the selection kernel
    int sel_impl = 1;               // 0 ticket, 1 automatic, 2 cluster wherever a group's CTAs fit one
    int sel_clu = 0;                // CTAs per group of the cluster selection (0: the ticket kernel runs)
    int sel_chunks_max = 0;         // the most selection CTAs a group needs
    int sel_sms = 1;                // SMs of the device (the selection plan's wave size: 4 CTAs each)
    // coalesce scratch: [2 (prefetch|urgent)][G][k][4], [2][G]
    int32_t* runs = nullptr;
    int32_t* nruns = nullptr;
    // attention scratch
    int4* att_items = nullptr;      // {group, part, first tile, n tiles}
    int32_t* att_first = nullptr;   // [G] first item of the group
    int32_t* att_count = nullptr;   // [G] items of the group
    int n_att_items = 0;
    int att_impl = 2;               // attention kernel: 0 register-direct loads, 1 TMA-staged persistent,
                                    // 2 group-split clusters (fused output; separate parts use 1)
    int att_cluster = 0;            // impl 2: CTAs per group asked for (0: automatic)
    int clu_S[2] = {1, 1};          // impl 2: CTAs per group, whole device and decode step
    bool clu_use[2] = {false, false};   // impl 2: clusters used (else the persistent kernel)
    bool att_pdl = true;            // impl 2: launched as a programmatic dependent of the kernel before it
    int att_part_cap = 0;           // work items the partial-result buffers hold
    // TMA-staged kernel: balanced per-CTA tile ranges cut into work items, one
    // plan for the whole device (standalone calls) and one for the decode step,
    // whose attention shares the device with a gather holding SMs of its own
    int tma_per_sm = 1;             // CTAs of the kernel resident per SM
    int clu_per_sm = 1;             // CTAs of the group-split cluster kernel resident per SM
    int n_sms = 1;
    int tma_ctas = 0;               // requested grid (0: fill the available SMs)
    struct TmaPlan {
        int grid = 0, n_items = 0;
        int4* items = nullptr;      // {group, part, first tile, tiles}
        int32_t* cta = nullptr;     // [grid + 1] first item of each CTA
        int32_t* first = nullptr;   // [G] first item of each group
        int32_t* count = nullptr;   // [G] items of each group
    } tma[2];
    long long att_wait_ns = 2000000000LL;   // limit of each mbarrier wait of the TMA-staged kernel
    int att_skip_tile = -1;         // >= 0: CTA 0 announces this tile without copying it (wait test)
    float* att_part_o = nullptr;    // [2][items][r][d]: two sets (launches side by side)
    float* att_part_ml = nullptr;   // [2][items][r][2]
    uint32_t* att_done = nullptr;   // [2][G]
    int32_t* status = nullptr;      // device status word
    // Gather launch shape and engine.  Default: the flat lane-load engine on 38
    // SM-exclusive CTAs of 1024 threads, 2 loads of K and of V in flight per lane.
    int gather_ctas = 38, gather_threads = 1024, gather_unroll = 2;
    int gather_engine = 3;          // 0: lane loads over runs, 1: TMA bulk copies, 3: flat lane loads over
                                    // entries, 4: copy engine (one cudaMemcpyAsync per run, issued by the host)
    std::vector<int64_t> h_off;     // host copies of the group offsets and candidate capacities (engine 4)
    std::vector<int32_t> h_Ccap;
    int32_t* h_runs = nullptr;      // pinned [G][k][4] run list read back for engine 4
    int32_t* h_nruns = nullptr;     // pinned [G]
    int gather_drivers = 0;         // TMA engine: driver warps (0: default)
    int gather_stages = 4;          // TMA engine: batches per driver (4 or 8)
    int gather_reserve_smem = 200 * 1024;   // flat engine: shared memory reserved per CTA (SM exclusivity)
    size_t scratch_bytes = 0;
    cudaStream_t s_compute = nullptr, s_prefetch = nullptr, s_urgent = nullptr;
    cudaStream_t s_urgent2 = nullptr;   // a chain step's odd layers' copies
    cudaStream_t s_hit = nullptr;       // a speculative step's hit passes (compute priority)
    // decode-step state
    int32_t* st_true = nullptr;     // [L][G][k]
    int32_t* st_pred = nullptr;     // [2][L][G][k]  predictions by step parity
    int32_t* st_miss = nullptr;     // [L][G][k]
    int32_t* st_miss_cnt = nullptr; // [L][G]
    int32_t* st_slot = nullptr;     // [L][G][k]
    int step_parity = 0;
    bool have_pred = false;
    // ordering events of the decode step; captured steps use their own set (an
    // event recorded inside a capture cannot be waited on outside it)
    struct EvSet {
        std::vector<cudaEvent_t> sel, attn, pref, urg, hit;   // hit: a split step's hit pass done
        std::vector<cudaEvent_t> rassign, rpref;   // resident mode, per layer: prefetch assigned / landed
        cudaEvent_t start = nullptr;
    } ev_eager, ev_graph;
    // optional per-launch timing of the decode step (kvo_profile)
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_pool;
    struct ProfRec { int kind; int ev; int layer; };
    std::vector<ProfRec> prof_recs;
    int prof_used = 0;
    // CUDA-graph replay of warm decode steps (one executable graph per step parity)
    bool use_graphs = false;
    cudaStream_t s_graph = nullptr;
    cudaEvent_t ev_gin = nullptr, ev_gout = nullptr;
    cudaGraphExec_t gexec[2] = {nullptr, nullptr};
    const void* gkey[2][6] = {};
    std::string err;
};

// kernel kinds reported by kvo_profile_read
enum ProfKind { PK_SELECT = 0, PK_DIFF = 1, PK_COALESCE = 2, PK_GATHER_PREFETCH = 3, PK_GATHER_URGENT = 4,
                PK_ATTENTION = 5, PK_RECON = 6, PK_COUNT = 7 };

// --------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t float_to_ordered(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Block-wide exclusive scan of one uint32 per thread (blockDim.x multiple of 32, <= 1024).
// `warp_sums` needs blockDim.x / 32 entries of shared memory.  Returns the
// exclusive prefix; *total receives the block total.  Contains __syncthreads().
// Release/acquire fence at device scope: orders the memory operations the
// calling thread has performed or observed (through a CTA barrier) before the
// ones after it, as the last-CTA ticket protocols need; lighter than the
// sequentially consistent fence of __threadfence().
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t s = lane < nw ? warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) warp_sums[lane] = s;   // inclusive warp prefix
    }
    __syncthreads();
    uint32_t base = wid ? warp_sums[wid - 1] : 0u;
    *total = warp_sums[nw - 1];
    __syncthreads();
    return base + x - v;
}

// ---------------------------------------------------------------- launchers
// Each returns cudaGetLastError() after the launch.
cudaError_t launch_landmarks(const Ctx& c, int layer, cudaStream_t s);
struct ResAssignArgs;   // resident_assign.cuh
// With `assign` (single-query steps only), the last CTA of each group also
// assigns the group's resident slots for the true index it selected.
// pdl: launched as a programmatic dependent of the kernel before it on the
// stream (waits for it before reading anything; standalone calls only).
cudaError_t launch_select(const Ctx& c, int layer, const void* q, const void* q_spec, int32_t* idx_true,
                          int32_t* idx_pred, cudaStream_t s, const ResAssignArgs* assign = nullptr,
                          bool pdl = false);
cudaError_t prepare_select_assign(const Ctx& c);
cudaError_t launch_index_diff(const Ctx& c, const int32_t* idx_true, const int32_t* idx_pred, int32_t* miss,
                              int32_t* miss_cnt, int32_t* slot, cudaStream_t s);
cudaError_t launch_coalesce(const Ctx& c, const int32_t* idx, const int32_t* cnt, int slot_base, int32_t* runs,
                            int32_t* nruns, cudaStream_t s);
cudaError_t launch_gather(const Ctx& c, int layer, int buf, const int32_t* runs, const int32_t* nruns,
                          cudaStream_t s);
cudaError_t launch_gather_tma(const Ctx& c, int layer, int buf, const int32_t* runs, const int32_t* nruns,
                              cudaStream_t s);
cudaError_t launch_gather_flat(const Ctx& c, int layer, int buf, const int32_t* idx, const int32_t* cnt, int slot_base,
                               cudaStream_t s, const int32_t* dslot = nullptr, int kv_mask = 3, bool alone = false);
cudaError_t launch_lowrank_k(const Ctx& c, int layer, int buf, const int32_t* idx, const int32_t* cnt, int slot_base,
                             const int32_t* dslot, cudaStream_t s);
cudaError_t prepare_lowrank();
cudaError_t launch_resident_assign(const Ctx& c, int layer, const int32_t* need, const int32_t* keep,
                                   int32_t* out_ids, int32_t* out_cnt, int32_t* out_dslot, int32_t* slot_of,
                                   int phase, cudaStream_t s, int max_fetch = -1, int32_t* hit_slot = nullptr,
                                   int32_t* hit_cnt = nullptr);
cudaError_t prepare_resident(const Ctx& c);
// The arguments launch_resident_assign passes (need, phase 0 or 1, ...), for
// the selection kernel's fused assignment.
ResAssignArgs resident_assign_args(const Ctx& c, int layer, const int32_t* need, const int32_t* keep,
                                   int32_t* out_ids, int32_t* out_cnt, int32_t* out_dslot, int32_t* slot_of,
                                   int phase, int max_fetch, int32_t* hit_slot, int32_t* hit_cnt);
// Optional for the TMA-staged kernel only: sp_cnt[g] limits the sparse part to
// the first sp_cnt[g] entries of the slot list; pdl launches it as a
// programmatic dependent of the kernel before it on the stream (it starts once
// that kernel's CTAs are all resident, and ends only after that kernel has
// completed).  scratch (0 or 1) picks one of the two sets of partial results
// and tickets the work-item kernels use, so two launches may run side by side.
cudaError_t launch_attention(const Ctx& c, int layer, int buf, const void* q, const void* q_spec, const int32_t* slot,
                             float* o, float* lse, float* o_spec, float* lse_spec, int fuse, cudaStream_t s,
                             bool in_step = false, const int32_t* sp_cnt = nullptr, bool pdl = false,
                             int scratch = 0);
// Attention over the first cnt[g] entries of a slot list, merged by lse with a
// prior part into (o, lse); merge_part_split(c) CTAs per group.
constexpr int MP_SPLIT_MAX = 8;
int merge_part_split(const Ctx& c);
cudaError_t launch_attn_merge_part(const Ctx& c, int buf, const void* q, const int32_t* slot, const int32_t* cnt,
                                   const float* prior_o, const float* prior_lse, float* o, float* lse,
                                   cudaStream_t s);
cudaError_t launch_merge_lse(const float* o1, const float* lse1, const float* o2, const float* lse2, float* o,
                             float* lse, int rows, int d, cudaStream_t s);
cudaError_t copy_landmarks_logical(const Ctx& c, int layer, void* dst, cudaStream_t s);
cudaError_t launch_ring_fill(const Ctx& c, int layer, const uint16_t* k_win, const uint16_t* v_win, cudaStream_t s);
cudaError_t launch_append(const Ctx& c, const void* k_new, const void* v_new, cudaStream_t s);

int gather_default_ctas(const Ctx& c);
// Raise the dynamic shared memory limits of the gather kernels (host call; done at init, never during capture).
cudaError_t prepare_gather_tma();
cudaError_t prepare_gather_flat();
cudaError_t prepare_attention(Ctx& c);

// Sets the message kvo_last_error(NULL) returns (context-free calls).
void set_last_error(const char* msg);

}  // namespace kvo
