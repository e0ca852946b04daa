// Host -> HBM gather driven by the Tensor Memory Accelerator (bulk copies).
//
// Same contract as gather_kernel ("PulseInfer and the I/O Problem Behind
// Long-Context Decoding", §2: coalesced gather of fragmented transfers;
// "DualDecoder: Accelerate Long Context LLM Inference by Predictive Prefetch",
// §5.4 / Fig. 11: ping-pong half as destination): every run of adjacent
// blocks is copied, K and V, from the host cache into its slots.
//
// Why TMA: a lane-load gather keeps ~1 MB of 16-byte zero-copy loads in flight
// to fill the host link, and each of those loads occupies its SM's load/store
// pipeline for the whole link round trip, which stalls HBM-bound kernels that
// share the SM.  Here one thread per warp ("driver") forms batches of up to
// TMA_STAGE_BYTES of run pieces, issues cp.async.bulk host -> shared memory
// completing on the stage's mbarrier, and once a batch has landed issues
// cp.async.bulk shared -> HBM stores (bulk groups).  TMA_STAGES - 1 batches per
// driver are in flight; a few dozen drivers fill the link while the SMs'
// load/store pipelines stay free.  Every mbarrier wait is bounded by the
// global timer: on expiry the driver records KVO_DEV_TIMEOUT and stops.
#include "kvo_internal.cuh"
#include "tma_ptx.cuh"

namespace kvo {

namespace {

struct Piece {
    unsigned long long src;   // host source (device-mapped)
    unsigned long long dst;   // global destination
    uint32_t soff;            // offset in the stage
    uint32_t bytes;
};

// Piece generator over one driver's runs: K then V of each run, cut into
// pieces of at most TMA_STAGE_BYTES.
struct RunCursor {
    const uint16_t *kh, *vh;
    const int64_t* g_off;
    const int32_t* g_C;
    const int4* runs;
    const int32_t* nruns;
    uint16_t *dk, *dv;
    int G, k, B, D;
    int64_t e, stride, total;
    int32_t* status;
    // current run
    bool have;
    int kv;
    int64_t src_el, dst_el;   // element offsets of the run (K and V share them)
    uint32_t bytes, off;

    __device__ bool next_run() {
        const int64_t blk = (int64_t)B * D;
        while (e < total) {
            const int bg = (int)(e / k);
            const int ri = (int)(e - (int64_t)bg * k);
            const int64_t cur = e;
            e += stride;
            if (ri >= nruns[bg]) continue;
            const int4 run = runs[cur];
            if (run.x < 0 || run.y < 1 || run.x + run.y > g_C[bg] || run.z < 0 || run.z + run.y > 2 * k) {
                atomicOr(status, KVO_DEV_BAD_SLOT);
                continue;
            }
            src_el = g_off[bg] + (int64_t)run.x * blk;
            dst_el = ((int64_t)bg * 2 * k + run.z) * blk;
            bytes = (uint32_t)(run.y * blk * 2);
            off = 0;
            kv = 0;
            have = true;
            return true;
        }
        have = false;
        return false;
    }
    // Next piece without consuming it.
    __device__ bool peek(const void** src, void** dst, uint32_t* n) {
        if (!have && !next_run()) return false;
        const uint16_t* s = kv ? vh : kh;
        uint16_t* d = kv ? dv : dk;
        *src = (const char*)(s + src_el) + off;
        *dst = (char*)(d + dst_el) + off;
        *n = min((uint32_t)TMA_STAGE_BYTES, bytes - off);
        return true;
    }
    __device__ void consume(uint32_t n) {
        off += n;
        if (off == bytes) {
            off = 0;
            if (kv == 0) kv = 1; else have = false;
        }
    }
};

}  // namespace

template <int TMA_STAGES>
__global__ void __launch_bounds__(64)
gather_tma_kernel(const uint16_t* __restrict__ kh, const uint16_t* __restrict__ vh, const int64_t* __restrict__ g_off,
                  const int32_t* __restrict__ g_C, const int4* __restrict__ runs, const int32_t* __restrict__ nruns,
                  uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, int G, int k, int B, int D, int n_drivers,
                  int32_t* __restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int driver = blockIdx.x * (blockDim.x >> 5) + w;
    if (lane != 0 || driver >= n_drivers) return;
    unsigned char* base = smem + (size_t)w * tma_driver_smem(TMA_STAGES);
    const uint32_t stage0 = smem_u32(base);
    Piece* plist = reinterpret_cast<Piece*>(base + TMA_STAGES * TMA_STAGE_BYTES);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(base + TMA_STAGES * TMA_STAGE_BYTES +
                                                 TMA_STAGES * TMA_MAX_PIECES * sizeof(Piece));
    int* pcount = reinterpret_cast<int*>(mbar + TMA_STAGES);
    for (int s = 0; s < TMA_STAGES; ++s) mbar_init(smem_u32(&mbar[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    RunCursor cur;
    cur.kh = kh; cur.vh = vh; cur.g_off = g_off; cur.g_C = g_C; cur.runs = runs; cur.nruns = nruns;
    cur.dk = dk; cur.dv = dv; cur.G = G; cur.k = k; cur.B = B; cur.D = D;
    cur.e = driver; cur.stride = n_drivers; cur.total = (int64_t)G * k; cur.status = status; cur.have = false;

    constexpr uint64_t kLimitNs = 2000000000ull;   // 2 s per wait
    long long formed = 0, stored = 0;
    bool failed = false;

    // Wait (bounded) for batch b to land, then store its pieces to HBM as one bulk group.
    auto store_batch = [&](long long b) -> bool {
        const int st = (int)(b % TMA_STAGES);
        const uint32_t parity = (uint32_t)((b / TMA_STAGES) & 1);
        const uint32_t mb = smem_u32(&mbar[st]);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(mb, parity)) {
            if (global_ns() - t0 > kLimitNs) {
                atomicOr(status, KVO_DEV_TIMEOUT);
                return false;
            }
        }
        const Piece* pl = plist + st * TMA_MAX_PIECES;
        const int n = pcount[st];
        const uint32_t sbase = stage0 + (uint32_t)st * TMA_STAGE_BYTES;
        for (int i = 0; i < n; ++i) bulk_store((void*)pl[i].dst, sbase + pl[i].soff, pl[i].bytes);
        bulk_commit();
        return true;
    };

    for (;;) {
        const int st = (int)(formed % TMA_STAGES);
        if (formed >= TMA_STAGES) bulk_wait_read_all();    // the stage's previous stores have read it
        Piece* pl = plist + st * TMA_MAX_PIECES;
        int n = 0;
        uint32_t used = 0;
        const void* src;
        void* dst;
        uint32_t nb;
        while (n < TMA_MAX_PIECES && cur.peek(&src, &dst, &nb)) {
            if (used + nb > (uint32_t)TMA_STAGE_BYTES) break;
            pl[n].src = (unsigned long long)src;
            pl[n].dst = (unsigned long long)dst;
            pl[n].soff = used;
            pl[n].bytes = nb;
            used += nb;
            ++n;
            cur.consume(nb);
        }
        if (n == 0) break;                                  // no work left for this driver
        pcount[st] = n;
        const uint32_t mb = smem_u32(&mbar[st]);
        const uint32_t sbase = stage0 + (uint32_t)st * TMA_STAGE_BYTES;
        mbar_expect_tx(mb, used);
        for (int i = 0; i < n; ++i) bulk_load(sbase + pl[i].soff, (const void*)pl[i].src, pl[i].bytes, mb);
        ++formed;
        if (formed - stored >= TMA_STAGES - 1) {
            if (!store_batch(stored)) { failed = true; break; }
            ++stored;
        }
    }
    while (!failed && stored < formed) {
        if (!store_batch(stored)) { failed = true; break; }
        ++stored;
    }
    bulk_wait_all();   // stores complete (and visible) before the driver exits
}

template <int STAGES>
static cudaError_t launch_tma_stages(const Ctx& c, int layer, int buf, const int32_t* runs, const int32_t* nruns,
                                     cudaStream_t s) {
    const int drivers = c.gather_drivers > 0 ? c.gather_drivers : 32;
    const int per_cta = STAGES >= 8 ? 1 : 2;
    const size_t smem = (size_t)per_cta * tma_driver_smem(STAGES);
    gather_tma_kernel<STAGES><<<(drivers + per_cta - 1) / per_cta, per_cta * 32, smem, s>>>(
        c.k_host[layer], c.v_host[layer], c.g_off, c.g_C, (const int4*)runs, nruns, c.buf_k(buf), c.buf_v(buf), c.G,
        c.k, c.B, c.d, drivers, c.status);
    return cudaGetLastError();
}

cudaError_t prepare_gather_tma() {
    cudaError_t e = cudaFuncSetAttribute(gather_tma_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(2 * tma_driver_smem(4)));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gather_tma_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tma_driver_smem(8));
}

cudaError_t launch_gather_tma(const Ctx& c, int layer, int buf, const int32_t* runs, const int32_t* nruns,
                              cudaStream_t s) {
    if (c.gather_stages >= 8) return launch_tma_stages<8>(c, layer, buf, runs, nruns, s);
    return launch_tma_stages<4>(c, layer, buf, runs, nruns, s);
}

}  // namespace kvo
