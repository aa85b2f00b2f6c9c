// k_tma.cu -- all-gather, gather and broadcast with the Tensor Memory Accelerator's bulk
// copies: "read once, write N times" without the per-thread store traffic.
//
// Each CTA streams tiles of its source blocks through a ring of shared-memory stages.
// One thread issues a bulk load (cp.async.bulk global -> shared, completing on an
// mbarrier) per tile and, once it has landed, one bulk store (cp.async.bulk shared ->
// global) per destination rank.  A stage is reloaded only after the stores that read it
// have finished reading (bulk async-group accounting), so loads for the next tiles are in
// flight while the current tile is being written N times.  The store streams go through
// the copy engine of the SM instead of the load/store unit, which throttles when every
// thread issues N stores per loaded vector.
//
// Every wait is bounded: a load that has not landed after kWaitNs makes the kernel record
// vTimeout in the status word, stop issuing, drain its own bulk operations and return.
#include <atomic>

#include "device.cuh"

namespace vc {

constexpr int kTmaStages = 4;
constexpr int kTmaTileBytes = 16 * 1024;
constexpr unsigned long long kWaitNs = 2000ull * 1000 * 1000;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}

__device__ __forceinline__ void bulk_load(void* smem, const void* gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(smem)), "l"(gmem), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void bulk_store(void* gmem, const void* smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gmem), "r"(smem_addr(smem)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// One CTA's share: tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... of the flat tile
// space of `nBlocks` source blocks of `blockBytes` each (block s = src[s] or the root's
// buffer), each tile written to ndst destinations at dst[d] + s * dstStride + offset.
struct TmaJob {
    const char* const* src;          // per block (rank) source pointer
    char* const* dst;                // destination pointers
    int ndst;
    int nBlocks;
    size_t blockBytes;               // bytes per block (a multiple of 16)
    size_t dstStride;                // destination offset between blocks
    int stages;                      // shared-memory tile stages (1..kTmaStages)
};

__device__ __forceinline__ void tile_of(const TmaJob& j, size_t tilesPerBlock, size_t t, int* s,
                                        size_t* off, uint32_t* bytes) {
    *s = (int)(t / tilesPerBlock);
    const size_t k = t - (size_t)(*s) * tilesPerBlock;
    *off = k * kTmaTileBytes;
    *bytes = (uint32_t)min((size_t)kTmaTileBytes, j.blockBytes - *off);
}

constexpr size_t tma_smem_bytes(int stages) {
    return (size_t)stages * kTmaTileBytes + (size_t)stages * sizeof(uint64_t);
}
constexpr size_t kTmaSmemBytes = tma_smem_bytes(kTmaStages);

__device__ void tma_fanout(const TmaJob& j, Status* st, volatile Status* stHost) {
    // dynamic shared memory: j.stages tiles, then one mbarrier per stage
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char (*stage)[kTmaTileBytes] = reinterpret_cast<unsigned char (*)[kTmaTileBytes]>(smem);
    const int S = j.stages;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (size_t)S * kTmaTileBytes);
    if (threadIdx.x != 0) return;
    const size_t tilesPerBlock = (j.blockBytes + kTmaTileBytes - 1) / kTmaTileBytes;
    const size_t nTiles = tilesPerBlock * (size_t)j.nBlocks;
    // this CTA's tiles: first = blockIdx.x, stride = gridDim.x; count
    const size_t first = blockIdx.x;
    if (first >= nTiles) return;
    const size_t mine = (nTiles - first + gridDim.x - 1) / gridDim.x;
    for (int b = 0; b < S; b++) mbar_init(&bar[b], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    auto issue_load = [&](size_t k) {
        const size_t t = first + k * gridDim.x;
        int s; size_t off; uint32_t bytes;
        tile_of(j, tilesPerBlock, t, &s, &off, &bytes);
        const int b = (int)(k % S);
        mbar_expect_tx(&bar[b], bytes);
        bulk_load(stage[b], j.src[s] + off, bytes, &bar[b]);
    };
    const size_t pre = min((size_t)S, mine);
    for (size_t k = 0; k < pre; k++) issue_load(k);
    size_t issued = pre;

    bool failed = false;
    size_t k = 0;
    for (; k < mine; k++) {
        const int b = (int)(k % S);
        const uint32_t parity = (uint32_t)((k / S) & 1);
        if (!mbar_try_wait(&bar[b], parity)) {
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&bar[b], parity)) {
                if (global_timer_ns() - t0 > kWaitNs) { failed = true; break; }
            }
        }
        if (failed) {
            report_error(st, stHost, vTimeout, blockIdx.x, 0, (unsigned)k);
            break;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const size_t t = first + k * gridDim.x;
        int s; size_t off; uint32_t bytes;
        tile_of(j, tilesPerBlock, t, &s, &off, &bytes);
        for (int d = 0; d < j.ndst; d++) bulk_store(j.dst[d] + (size_t)s * j.dstStride + off, stage[b], bytes);
        bulk_commit();
        // Refill a stage once the stores that read it are done: with one stage, this
        // tile's own (then tile k + 1 goes in); otherwise the previous tile's, so this
        // tile's stores stay in flight (then tile k - 1 + S goes in).
        if (S == 1) {
            if (k + 1 < mine) {
                bulk_wait_read<0>();
                issue_load(k + 1);
                issued++;
            }
        } else if (k >= 1 && k - 1 + S < mine) {
            bulk_wait_read<1>();
            issue_load(k - 1 + S);
            issued++;
        }
    }
    bulk_wait_all();
    if (failed) {
        // Loads still in flight target shared memory that is released when the CTA exits:
        // give each a bounded wait before returning.
        for (size_t q = k; q < issued; q++) {
            const int b = (int)(q % S);
            const uint32_t parity = (uint32_t)((q / S) & 1);
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&bar[b], parity) && global_timer_ns() - t0 < kWaitNs) {
            }
        }
    }
}

// All-gather (outRoot < 0) or gather (outRoot = root): blocks s = send[s], sc elements,
// land at recv[r] + s * sc.  Broadcast: one block send[root] to every recv[r].
__global__ void __launch_bounds__(32) k_fanout_tma(const __grid_constant__ OnePassArgs a, int esz, int isBroadcast,
                                                  int stages, Status* st, Status* stHost) {
    pdl_begin();
    TmaJob j;
    j.stages = stages;
    const char* const* sends = (const char* const*)a.send;
    j.dst = a.outRoot >= 0 ? (char* const*)&a.recv[a.outRoot] : (char* const*)a.recv;
    j.ndst = a.outRoot >= 0 ? 1 : a.nRanks;
    if (isBroadcast) {
        j.src = &sends[a.root];
        j.nBlocks = 1;
        j.blockBytes = a.count * (size_t)esz;
        j.dstStride = 0;
    } else {
        j.src = sends;
        j.nBlocks = a.nRanks;
        j.blockBytes = a.count * (size_t)esz;
        j.dstStride = j.blockBytes;
    }
    tma_fanout(j, st, stHost);
}

cudaError_t launch_fanout_tma(const OnePassArgs& a, int elemSize, bool broadcast, int grid, int stages,
                              Status* st, volatile Status* stHost, cudaStream_t s) {
    if (stages < 1 || stages > kTmaStages) return cudaErrorInvalidValue;
    // The shared-memory limit is an attribute of the function on each device: set it once
    // per device (bit d of the mask).
    static std::atomic<unsigned long long> attrSet{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attrSet.load() & bit)) {
        e = cudaFuncSetAttribute(k_fanout_tma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmaSmemBytes);
        if (e != cudaSuccess) return e;
        attrSet.fetch_or(bit);
    }
    return pdl_launch(k_fanout_tma, grid, 32, tma_smem_bytes(stages), s, a, elemSize, broadcast ? 1 : 0,
                      stages, st, (Status*)stHost);
}

}  // namespace vc
