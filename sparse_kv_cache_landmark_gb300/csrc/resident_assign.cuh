// Assignment of a (layer, group)'s resident slots, shared by the assignment
// kernel and the selection kernel that runs it in each group's last CTA.
//
// Cross-step delta prefetch: per (layer, group) a GPU-resident block set of 2k
// slots outlives the decode step, and each step fetches only the blocks it
// does not already hold ("NeuroPrefetcher: Storage-Aware Sparse LLM Inference
// via Delta Prefetching", title; "DualDecoder: Accelerate Long Context LLM
// Inference by Predictive Prefetch", §5.2 / Fig. 18: the true index's misses
// are fetched urgently before attention).
//
// Rule (the pages give none; the plainest one that keeps every copy
// destination decided before the copy starts): the blocks of the `need` list
// already resident stay in their slots; the missing ones, in ascending id
// order, take the reusable slots in ascending slot order, a slot being
// reusable when it is empty or holds a block in neither `need` nor `keep`.
// The decode step calls it twice per layer: urgent (need = true index, keep =
// the prediction fetched for this step) and, after attention, prefetch (need
// = the prediction for the next step, keep = the true index).  With 2k slots
// neither call runs out of reusable slots.
//
// Outputs: the fetched blocks (ascending ids) with their destination slots and
// count, (optional) the slot of every need entry after the update, and
// (optional) the slots of the need entries that were resident already, in need
// order, with their count (the blocks attention may read before the fetch).
// max_fetch >= 0 admits only the max_fetch missing blocks with the lowest ids
// (a cap on host bytes, used for the prefetch phase only; "PulseInfer and the
// I/O Problem Behind Long-Context Decoding", §2: I/O-adaptive offloading
// admission, given there without a rule).
//
// Speculation accounting (pfbit, stat; nullable): a slot filled by the
// prefetch phase is marked until a true index uses it; stat[0] counts the
// blocks the prefetch phase fetched, stat[1] the marked blocks an urgent phase
// found in its true index -- a speculative fetch that saved an urgent one.
//
// Speculation policy (pol, ticket; nullable): pol = {on, steps, fetched,
// used, rest} of the layer's current window.  A used prefetch saves an urgent
// fetch, an unused one costs a fetch, so prefetching pays while more than half
// of the prefetched blocks are used.  The last group of an urgent phase (atomic
// ticket over the n_groups groups) closes a window of KVO_SPEC_WINDOW steps: a
// layer whose window failed that test stops prefetching for `rest` steps and
// then tries again; rest starts at KVO_SPEC_REST, doubles with every failed try
// (up to KVO_SPEC_REST_MAX) and returns to KVO_SPEC_REST after a window that
// paid.  A prefetch phase of a layer that is off fetches nothing.  Both phases
// of a layer run in stream order, so the state needs no other synchronisation.
#pragma once
#include "kvo_internal.cuh"

namespace kvo {

#define KVO_SPEC_WINDOW 4ull
#define KVO_SPEC_REST 32ull
#define KVO_SPEC_REST_MAX 1024ull

struct ResAssignArgs {
    const int32_t* need;       // [G][k] ascending ids
    const int32_t* keep;       // [G][k] or null
    int32_t* map;              // [G][Ccap] block -> slot (-1: not resident), this layer
    int32_t* slots;            // [G][cap] slot -> block (-1: empty)
    const int32_t* g_C;        // [G] host-resident blocks
    int32_t* out_ids;          // [G][k] fetched blocks
    int32_t* out_cnt;          // [G]
    int32_t* out_dslot;        // [G][k] their slots
    int32_t* slot_of;          // [G][k] or null: slot of every need entry
    int32_t* hit_slot;         // [G][k] or null: slots of the entries resident before
    int32_t* hit_cnt;          // [G] or null
    unsigned long long* fetched;
    int k, cap, Ccap, max_fetch;
    uint8_t* pfbit;
    unsigned long long* stat;
    int phase;                 // 0 urgent, 1 prefetch
    unsigned long long* pol;
    uint32_t* ticket;
    int n_groups;
    int32_t* status;
};

// shared-memory ints the routine needs: need, keep, missing ids (k each) and
// reusable slots (cap = 2k)
__host__ __device__ constexpr size_t res_assign_ints(int k) { return 5 * (size_t)k; }

__device__ __forceinline__ bool sorted_contains(const int32_t* a, int n, int32_t x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo < n && a[lo] == x;
}

// Group g's assignment by the whole CTA (any multiple of 32 threads): rs holds
// res_assign_ints(k) ints of shared memory, warp_sums 32 words, s_tot one.
__device__ __forceinline__ void resident_assign_group(const ResAssignArgs& a, int g, int32_t* rs, uint32_t* warp_sums,
                                                      uint32_t* s_tot) {

    const int tid = threadIdx.x, nt = blockDim.x;
    const int k = a.k, cap = a.cap, Ccap = a.Ccap, phase = a.phase;
    int max_fetch = a.max_fetch;
    const int32_t* need = a.need;
    const int32_t* keep = a.keep;
    uint8_t* pfbit = a.pfbit;
    unsigned long long* stat = a.stat;
    unsigned long long* pol = a.pol;
    int32_t* s_need = rs;                  // [k]
    int32_t* s_keep = s_need + k;          // [k]
    int32_t* s_ev = s_keep + k;            // [cap] reusable slots in ascending order
    int32_t* s_mid = s_ev + cap;           // [k] missing ids, ascending
    const int C = min(a.g_C[g], Ccap);
    int32_t* mg = a.map + (int64_t)g * Ccap;
    int32_t* sg = a.slots + (int64_t)g * cap;
    uint8_t* pg = pfbit ? pfbit + (int64_t)g * cap : nullptr;
    int bad = 0;
    for (int i = tid; i < k; i += nt) {
        s_need[i] = need[(int64_t)g * k + i];
        s_keep[i] = keep ? keep[(int64_t)g * k + i] : -1;
    }
    __syncthreads();
    const int nk = keep ? k : 0;

    // 1. reusable slots (each thread scans a contiguous chunk)
    const int per = (cap + nt - 1) / nt;
    const int s0 = min(cap, tid * per), s1 = min(cap, s0 + per);
    uint32_t nev = 0;
    for (int s = s0; s < s1; ++s) {
        const int32_t b = sg[s];
        nev += (b < 0 || (!sorted_contains(s_need, k, b) && !sorted_contains(s_keep, nk, b))) ? 1u : 0u;
    }
    uint32_t base = block_exclusive_scan(nev, warp_sums, s_tot);
    const uint32_t n_ev = *s_tot;
    for (int s = s0; s < s1; ++s) {
        const int32_t b = sg[s];
        if (b < 0 || (!sorted_contains(s_need, k, b) && !sorted_contains(s_keep, nk, b))) s_ev[base++] = s;
    }

    // 2. missing need entries (contiguous chunks keep the ascending order)
    const int pk = (k + nt - 1) / nt;
    const int i0 = min(k, tid * pk), i1 = min(k, i0 + pk);
    uint32_t nm = 0, used = 0;
    for (int i = i0; i < i1; ++i) {
        const int32_t x = s_need[i];
        if (x < 0 || x >= C) { bad |= KVO_DEV_BAD_BLOCK_ID; continue; }
        const int32_t sx = mg[x];
        nm += sx < 0 ? 1u : 0u;
        // a true index meeting a block the prefetch phase fetched (need entries
        // are distinct, so no two threads touch one slot)
        if (phase == 0 && pg && sx >= 0 && pg[sx]) {
            ++used;
            pg[sx] = 0;
        }
    }
    if (stat && used) atomicAdd(stat + 1, (unsigned long long)used);
    if (pol && used) atomicAdd(pol + 3, (unsigned long long)used);
    base = block_exclusive_scan(nm, warp_sums, s_tot);
    const uint32_t n_miss = *s_tot;
    for (int i = i0; i < i1; ++i) {
        const int32_t x = s_need[i];
        if (x >= 0 && x < C && mg[x] < 0) s_mid[base++] = x;
    }
    if (a.hit_slot) {   // entries resident before the update keep their slots through it
        uint32_t nh = 0;
        for (int i = i0; i < i1; ++i) {
            const int32_t x = s_need[i];
            nh += (x >= 0 && x < C && mg[x] >= 0) ? 1u : 0u;
        }
        uint32_t hb = block_exclusive_scan(nh, warp_sums, s_tot);
        for (int i = i0; i < i1; ++i) {
            const int32_t x = s_need[i];
            if (x >= 0 && x < C && mg[x] >= 0) a.hit_slot[(int64_t)g * k + hb++] = mg[x];
        }
        if (tid == 0) a.hit_cnt[g] = (int32_t)*s_tot;
    }
    __syncthreads();
    // admission: at most max_fetch fetches (lowest ids first) when max_fetch >= 0;
    // none when the speculation policy has switched the layer's prefetch off
    if (phase == 1 && pol && *(volatile unsigned long long*)pol == 0ull) max_fetch = 0;
    const uint32_t wanted = max_fetch >= 0 ? min(n_miss, (uint32_t)max_fetch) : n_miss;
    const int n_fetch = (int)min(wanted, n_ev);
    if (wanted > n_ev && tid == 0) bad |= KVO_DEV_BAD_COUNT;

    // 3. evict the old occupants, then map the fetched blocks
    for (int j = tid; j < n_fetch; j += nt) {
        const int32_t old = sg[s_ev[j]];
        if (old >= 0 && old < Ccap) mg[old] = -1;
    }
    __syncthreads();
    for (int j = tid; j < n_fetch; j += nt) {
        const int32_t x = s_mid[j], s = s_ev[j];
        mg[x] = s;
        sg[s] = x;
        if (pg) pg[s] = phase == 1 ? 1 : 0;
        a.out_ids[(int64_t)g * k + j] = x;
        a.out_dslot[(int64_t)g * k + j] = s;
    }
    __syncthreads();
    if (a.slot_of) {
        for (int i = tid; i < k; i += nt) {
            const int32_t x = s_need[i];
            int32_t s = (x >= 0 && x < C) ? mg[x] : -1;
            if (s < 0) s = 0;                      // only after a reported error
            a.slot_of[(int64_t)g * k + i] = s;
        }
    }
    if (tid == 0) {
        a.out_cnt[g] = n_fetch;
        if (a.fetched && n_fetch) atomicAdd(a.fetched, (unsigned long long)n_fetch);
        if (phase == 1 && stat && n_fetch) atomicAdd(stat, (unsigned long long)n_fetch);
        if (phase == 1 && pol && n_fetch) atomicAdd(pol + 2, (unsigned long long)n_fetch);
    }
    if (phase == 0 && pol) {
        // the CTA's counts reach thread 0 through the barrier; its release fence
        // orders them before the ticket, the last CTA's acquire fence after it
        __syncthreads();
        if (tid == 0) {
            fence_acq_rel_gpu();
            if (atomicAdd(a.ticket, 1u) + 1 == (uint32_t)a.n_groups) {
                fence_acq_rel_gpu();
                volatile unsigned long long* v = pol;
                const unsigned long long steps = v[1] + 1;
                const unsigned long long rest = v[4] ? v[4] : KVO_SPEC_REST;
                if (v[0]) {
                    if (steps >= KVO_SPEC_WINDOW) {
                        if (v[2] > 0 && 2 * v[3] < v[2]) {
                            v[0] = 0;                                   // off for `rest` steps
                        } else {
                            v[4] = KVO_SPEC_REST;                       // a window that paid
                        }
                        v[1] = 0; v[2] = 0; v[3] = 0;
                    } else {
                        v[1] = steps;
                    }
                } else if (steps >= rest) {
                    v[0] = 1; v[1] = 0; v[2] = 0; v[3] = 0;             // try again; rest doubles if it fails
                    v[4] = rest * 2 < KVO_SPEC_REST_MAX ? rest * 2 : KVO_SPEC_REST_MAX;
                } else {
                    v[1] = steps;
                }
                *a.ticket = 0u;
            }
        }
    }
    if (bad) atomicOr(a.status, bad);
}

}  // namespace kvo
