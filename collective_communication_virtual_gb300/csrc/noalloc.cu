// noalloc.cu -- the staged ring all-reduce for callers that cannot allocate memory.
//
// Some callers cannot call cudaMalloc: allocators and memory-pool callbacks that must not
// recurse into the allocator, and runtimes that hand out all device memory themselves
// ahead of time and own every byte of it.  vcommInit allocates (its status
// words, and the ring FIFOs on first use), so those callers cannot use a communicator.
// vAllReduceNoAlloc gives them the ring all-reduce without one: its FIFOs and control
// words live in a fixed array compiled into this library.
//
// The array is a file-scope __device__ variable.  Host code cannot use its name as a
// device address (on the host the name is only a stand-in), so the first call on each
// device looks the real address up with cudaGetSymbolAddress while that device is
// current and keeps it.  Every GPU that loads the library holds the array until the
// process exits.  A cudaDeviceReset unloads the module and with it the array; every call
// therefore first checks, with cudaPointerGetAttributes, that the kept address is still a
// device allocation of the current context, and looks it up again if not.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kCtrlRegion = 64 * 1024;                 // status + per-(channel, rank) control
constexpr size_t kFifoRegion = 8u << 20;                  // FIFO slots
constexpr size_t kScratchBytes = kCtrlRegion + kFifoRegion;
// Data bytes per chunk (4 slots): 64 KiB for Simple; 32 KiB for LL and LL128, whose slots
// take more FIFO bytes than they carry.  Every protocol then fits 64 (channel, rank) FIFOs.
constexpr size_t kChunkBytes = 64 * 1024;
constexpr size_t kChunkBytesFlagged = 32 * 1024;
constexpr int kMaxDevices = 64;
constexpr unsigned long long kTimeoutNs = 2000ull * 1000 * 1000;

// Layout: [0, 16) device status word, [64, 68) device abort word, [128, 132) a word that
// stays zero and stands in for the host abort flag, [256, 256 + 256 * pairs) control
// blocks, [kCtrlRegion, kScratchBytes) FIFOs.
static __device__ __align__(256) unsigned char g_ringScratch[kScratchBytes];

std::mutex g_setupMutex;
unsigned char* g_scratchAddr[kMaxDevices];                // device address per device, set once

size_t elem_size(int dt) {
    switch (dt) {
    case vFloat32: case vInt32: return 4;
    case vFloat16: case vBFloat16: return 2;
    default: return 0;
    }
}

// Per-device set-up: the scratch array's device address, looked up with the device current
// (again if a device reset has invalidated the kept one).
cudaError_t scratch_address(int dev, unsigned char** out) {
    std::lock_guard<std::mutex> lock(g_setupMutex);
    if (g_scratchAddr[dev]) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, g_scratchAddr[dev]) != cudaSuccess || attr.type != cudaMemoryTypeDevice ||
            attr.device != dev) {
            cudaGetLastError();
            g_scratchAddr[dev] = nullptr;
        }
    }
    if (!g_scratchAddr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_ringScratch);
        if (e != cudaSuccess) return e;
        g_scratchAddr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratchAddr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" vResult_t vAllReduceNoAlloc(const void* const* sendbuffs, void* const* recvbuffs,
                                       size_t count, vDataType_t datatype, vRedOp_t op, int nRanks,
                                       int nChannels, vProto_t protocol, cudaStream_t stream) {
    if (nRanks < 2 || nRanks > VCOMM_MAX_RANKS || nChannels < 1 || nChannels > VCOMM_MAX_CHANNELS)
        return vInvalidArgument;
    if (protocol != vProtoSimple && protocol != vProtoLL && protocol != vProtoLL128) return vInvalidArgument;
    if (op < vSum || op > vMax) return vInvalidArgument;
    const size_t esz = elem_size(datatype);
    if (esz == 0 || !sendbuffs || !recvbuffs) return vInvalidArgument;
    if (count > ((size_t)1 << 62) / ((size_t)nRanks * esz)) return vInvalidArgument;

    vPlanRequest_t q = {};
    q.nRanks = nRanks;
    q.nChannels = nChannels;
    q.proto = protocol;
    q.algo = vAlgoRing;
    q.coll = vCollAllReduce;
    q.datatype = datatype;
    q.count = count;
    q.chunkBytes = protocol == vProtoSimple ? kChunkBytes : kChunkBytesFlagged;
    bool a16 = true;
    for (int r = 0; r < nRanks; r++) {
        const uintptr_t s = (uintptr_t)sendbuffs[r], d = (uintptr_t)recvbuffs[r];
        if (!s || !d || (s % esz) != 0 || (d % esz) != 0) return vInvalidArgument;
        a16 = a16 && (s % 16) == 0 && (d % 16) == 0;
    }
    q.aligned16 = a16 ? 1 : 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return vUnhandledCudaError;
    int sm = 0;
    if (cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return vUnhandledCudaError;
    q.smCount = sm;
    vPlanInfo_t p;
    vResult_t r = vPlanCompute(&q, &p);
    if (r != vSuccess) return r;
    // The array holds at most this many (channel, rank) FIFOs; larger rings are refused.
    const size_t pairs = (size_t)nRanks * nChannels;
    if (pairs * p.fifoBytes > kFifoRegion || 256 + pairs * vc::kCtrlStride * 8 > kCtrlRegion)
        return vInvalidArgument;
    if (count == 0) return vSuccess;

    int maxCtas = 0;
    if (vc::ring_max_coresident(datatype, op, datatype, (vProto_t)p.proto, p.threadsPerCta, sm, &maxCtas) !=
        cudaSuccess)
        return vUnhandledCudaError;
    if (p.gridCtas > maxCtas) return vInvalidUsage;

    unsigned char* base = nullptr;
    if (scratch_address(dev, &base) != cudaSuccess) return vUnhandledCudaError;

    // The array keeps the previous call's contents: clear the status, control words and
    // the FIFO slots this call uses, so counters and flags start from zero.
    if (cudaMemsetAsync(base, 0, 256 + pairs * vc::kCtrlStride * 8, stream) != cudaSuccess ||
        cudaMemsetAsync(base + kCtrlRegion, 0, pairs * p.fifoBytes, stream) != cudaSuccess)
        return vUnhandledCudaError;

    vc::RingArgs a = {};
    for (int i = 0; i < nRanks; i++) {
        a.send[i] = sendbuffs[i];
        a.recv[i] = recvbuffs[i];
    }
    a.nRanks = nRanks;
    a.nChannels = nChannels;
    a.coll = vCollAllReduce;
    a.op = op;
    a.root = 0;
    a.aligned = p.vectorized;
    a.hasScale = 0;
    a.scale = 1.0f;
    a.count = count;
    a.blockElems = p.blockElems;
    a.chanElems = p.channelElems;
    a.chunkElems = p.chunkElems;
    a.slotElems = p.slotPayloadElems;
    a.slotBytes = p.slotBytes;
    a.fifo = reinterpret_cast<char*>(base + kCtrlRegion);
    a.ctrl = reinterpret_cast<unsigned long long*>(base + 256);
    a.epochHi = 1ull << 32;                   // counters were just cleared: one epoch suffices
    a.llEpoch = 1u << 24;
    a.timeoutNs = kTimeoutNs;
    a.abortHost = reinterpret_cast<volatile unsigned int*>(base + 128);
    a.abortDev = reinterpret_cast<unsigned int*>(base + 64);
    a.status = reinterpret_cast<vc::Status*>(base);
    a.statusHost = nullptr;
    a.testStallRank = -1;
    a.testJitterNs = 0;
    a.testBadFlagRank = -1;
    const cudaError_t e =
        vc::launch_ring(a, datatype, op, datatype, (vProto_t)p.proto, p.gridCtas, p.threadsPerCta, stream);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        return vInvalidUsage;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return vUnhandledCudaError;
    }
    return vSuccess;
}
