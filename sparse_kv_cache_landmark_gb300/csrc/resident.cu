// Resident slot assignment as its own kernel: one CTA per group running the
// routine of resident_assign.cuh (the rule, outputs and speculation policy are
// described there).
#include "resident_assign.cuh"

namespace kvo {

constexpr int RES_THREADS = 512;

__global__ void __launch_bounds__(RES_THREADS) resident_assign_kernel(const ResAssignArgs a) {
    extern __shared__ __align__(16) int32_t rs[];
    __shared__ uint32_t warp_sums[32];
    __shared__ uint32_t s_tot;
    resident_assign_group(a, blockIdx.x, rs, warp_sums, &s_tot);
}

static size_t res_smem(const Ctx& c) { return sizeof(int32_t) * res_assign_ints(c.k); }

cudaError_t prepare_resident(const Ctx& c) {
    return cudaFuncSetAttribute(resident_assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)res_smem(c));
}

ResAssignArgs resident_assign_args(const Ctx& c, int layer, const int32_t* need, const int32_t* keep,
                                   int32_t* out_ids, int32_t* out_cnt, int32_t* out_dslot, int32_t* slot_of,
                                   int phase, int max_fetch, int32_t* hit_slot, int32_t* hit_cnt) {
    const int cap = 2 * c.k;
    ResAssignArgs a;
    a.need = need; a.keep = keep;
    a.map = c.res_map + (size_t)layer * c.G * c.Cmax;
    a.slots = c.res_slots + (size_t)layer * c.G * cap;
    a.g_C = c.g_C;
    a.out_ids = out_ids; a.out_cnt = out_cnt; a.out_dslot = out_dslot; a.slot_of = slot_of;
    a.hit_slot = hit_slot; a.hit_cnt = hit_cnt;
    a.fetched = c.res_fetched + phase;
    a.k = c.k; a.cap = cap; a.Ccap = c.Cmax; a.max_fetch = max_fetch;
    a.pfbit = c.res_pfbit ? c.res_pfbit + (size_t)layer * c.G * cap : nullptr;
    a.stat = c.res_stat ? c.res_stat + 2 * (size_t)layer : nullptr;
    a.phase = phase;
    a.pol = (c.spec_policy == 1 && c.res_pol) ? c.res_pol + 8 * (size_t)layer : nullptr;
    a.ticket = c.res_pol_ticket ? c.res_pol_ticket + layer : nullptr;
    a.n_groups = c.G;
    a.status = c.status;
    return a;
}

// phase 0: urgent (counts into res_fetched[0]), 1: prefetch (res_fetched[1])
cudaError_t launch_resident_assign(const Ctx& c, int layer, const int32_t* need, const int32_t* keep,
                                   int32_t* out_ids, int32_t* out_cnt, int32_t* out_dslot, int32_t* slot_of,
                                   int phase, cudaStream_t s, int max_fetch, int32_t* hit_slot, int32_t* hit_cnt) {
    resident_assign_kernel<<<c.G, RES_THREADS, res_smem(c), s>>>(resident_assign_args(
        c, layer, need, keep, out_ids, out_cnt, out_dslot, slot_of, phase, max_fetch, hit_slot, hit_cnt));
    return cudaGetLastError();
}

}  // namespace kvo
