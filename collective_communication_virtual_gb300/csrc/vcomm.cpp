// vcomm.cpp -- the C ABI of libvcomm: communicator lifecycle, argument checks, planning
// and launch of the collectives on the caller's stream.
//
// Checks follow ncclEnqueueCheck / taskAppend (NCCL book chapter 6): a bad communicator
// or argument returns vInvalidArgument without enqueuing anything; count == 0 returns
// vSuccess at once; a sticky asynchronous error makes every later call return it
// (NCCL book section 2.1, asyncResult).  The communicator carries start/end magic words
// like ncclComm so a destroyed or foreign handle is refused.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <new>
#include <vector>

#include "internal.h"

namespace vc {
bool& pdl_enabled() {
    thread_local bool on = true;      // set from the communicator of the call being launched
    return on;
}
}  // namespace vc

namespace {

constexpr unsigned long long kMagic = 0x76636F6D6D763031ull;   // "vcommv01"
constexpr int kTrackedStreams = 16;

// The last launch that used communicator memory on one stream.
struct StreamEvent {
    cudaStream_t stream;
    cudaEvent_t event;
    bool recorded;
};

struct Config {
    vAlgo_t algo = vAlgoAuto;
    size_t chunkBytes = 0;           // 0: planner default
    int timeoutMs = 2000;
    bool debug = false;
    bool bulkCopy = false;           // TMA bulk copies for the fan-out copies (opt-in)
    bool persistentGrid = false;     // one-pass grids of one resident wave (A/B switch)
    bool pdl = true;                 // programmatic dependent launch of the one-pass kernels
};

// One call recorded between vcommGroupStart and vcommGroupEnd.
struct GroupRec {
    bool fusable = false;            // a one-pass all-reduce (fused with its peers)
    std::vector<const void*> send;
    std::vector<void*> recv;
    size_t count = 0;
    vDataType_t dt = vFloat32;
    vRedOp_t op = vSum;
    cudaStream_t stream = nullptr;
    int vecBytes = 0;
    size_t blockElems = 0;
    std::function<vResult_t()> launch; // every other call
};

}  // namespace

struct vcomm {
    unsigned long long startMagic;
    int nRanks;
    int nChannels;
    vProto_t proto;
    Config cfg;
    int device;
    int smCount;
    size_t l2Bytes;
    int cooperative;
    // status: device copy decides the first error; pinned mirror for the host
    vc::Status* statusDev;
    vc::Status* statusHost;          // pinned, mapped
    vc::Status* statusHostDev;       // its device address
    unsigned int* abortHost;         // pinned, mapped
    unsigned int* abortHostDev;
    unsigned int* abortDev;
    vResult_t hostError;             // sticky error found on the host side
    // ring staging
    char* fifo;
    size_t fifoCap;
    unsigned long long* ctrl;
    unsigned int epoch;
    int testStallRank;
    unsigned int testJitterNs;
    int testBadFlagRank;
    StreamEvent tracked[kTrackedStreams];   // per stream; reused round-robin when full
    unsigned int trackedNext;
    // group batching
    int groupDepth;
    std::vector<GroupRec>* group;
    vc::GroupArgs* groupArgs;        // host copy of a batch's parameter block
    unsigned int* tileCounters;      // variable all-to-all tile counters (device)
    unsigned int tileCounterSeq;     // eager calls: next pair of the rotating set
    unsigned int capturedCounterSeq; // captured calls: next pair of the captured set
    unsigned long long endMagic;
};

namespace {

size_t elem_size(int dt) {
    switch (dt) {
    case vFloat32: case vInt32: return 4;
    case vFloat16: case vBFloat16: return 2;
    default: return 0;
    }
}

// An NVTX range around every entry point that enqueues work, named after it, for Nsight
// Systems and other NVTX-aware tools (NCCL marks its API the same way, NCCL book section
// 2.1).  Header-only NVTX: with no tool attached a range costs a few nanoseconds.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

bool comm_ok(const vcomm* c) {
    return c != nullptr && c->startMagic == kMagic && c->endMagic == kMagic;
}

// Make the communicator's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    // Also selects the communicator's launch mode for this thread's launches.
    explicit DeviceGuard(const vcomm* c) : DeviceGuard(c->device) { vc::pdl_enabled() = c->cfg.pdl; }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

vResult_t sticky(vcomm* c) {
    if (c->hostError != vSuccess) return c->hostError;
    const unsigned code = *(volatile unsigned*)&c->statusHost->code;
    return (vResult_t)code;
}

vResult_t cuda_fail(vcomm* c, cudaError_t e, const char* what) {
    if (c && c->cfg.debug) std::fprintf(stderr, "vcomm: %s failed: %s\n", what, cudaGetErrorString(e));
    cudaGetLastError();     // clear a non-sticky launch error
    return vUnhandledCudaError;
}

void read_env(Config* cfg) {
    if (const char* s = std::getenv("VCOMM_ALGO")) {
        if (!std::strcmp(s, "onepass")) cfg->algo = vAlgoOnePass;
        else if (!std::strcmp(s, "ring")) cfg->algo = vAlgoRing;
        else if (!std::strcmp(s, "tree")) cfg->algo = vAlgoTree;
        else cfg->algo = vAlgoAuto;
    }
    if (const char* s = std::getenv("VCOMM_CHUNK_BYTES")) {
        const unsigned long long v = std::strtoull(s, nullptr, 0);
        if (v >= 4096 && v <= (64ull << 20) && (v & (v - 1)) == 0) cfg->chunkBytes = (size_t)v;
    }
    if (const char* s = std::getenv("VCOMM_TIMEOUT_MS")) {
        const long v = std::strtol(s, nullptr, 0);
        if (v >= 1 && v <= 3600 * 1000) cfg->timeoutMs = (int)v;
    }
    if (const char* s = std::getenv("VCOMM_DEBUG")) cfg->debug = !std::strcmp(s, "INFO");
    if (const char* s = std::getenv("VCOMM_COPY_TMA")) cfg->bulkCopy = !std::strcmp(s, "1");
    if (const char* s = std::getenv("VCOMM_GRID")) cfg->persistentGrid = !std::strcmp(s, "persistent");
    if (const char* s = std::getenv("VCOMM_PDL")) cfg->pdl = std::strcmp(s, "0") != 0;
}

void free_comm(vcomm* c) {
    delete c->group;
    delete c->groupArgs;
    for (auto& t : c->tracked)
        if (t.event) cudaEventDestroy(t.event);
    if (c->fifo) cudaFree(c->fifo);
    if (c->ctrl) cudaFree(c->ctrl);
    if (c->statusDev) cudaFree(c->statusDev);
    if (c->abortDev) cudaFree(c->abortDev);
    if (c->tileCounters) cudaFree(c->tileCounters);
    if (c->statusHost) cudaFreeHost(c->statusHost);
    if (c->abortHost) cudaFreeHost(c->abortHost);
    c->startMagic = c->endMagic = 0;
    delete c;
}

const char* coll_name(int coll) {
    static const char* n[] = {"AllReduce", "ReduceScatter", "AllGather", "Broadcast", "AllToAll",
                              "AllToAllv", "Reduce", "Gather", "Scatter"};
    return (coll >= 0 && coll <= 8) ? n[coll] : "?";
}

void debug_plan(const vcomm* c, int coll, size_t count, int dt, const vPlanInfo_t& p) {
    if (!c->cfg.debug) return;
    std::fprintf(stderr,
                 "vcomm INFO %s count=%zu dt=%d N=%d algo=%s proto=%d channels=%d ctas/ch=%d grid=%d "
                 "threads=%d vec=%d B=%zu Lc=%zu chunk=%zu slotElems=%zu slotBytes=%zu\n",
                 coll_name(coll), count, dt, c->nRanks, p.algo == vAlgoRing ? "ring" : "onepass", p.proto,
                 p.nChannels, p.ctasPerChannel, p.gridCtas, p.threadsPerCta, p.vectorized, p.blockElems,
                 p.channelElems, p.chunkElems, p.slotPayloadElems, p.slotBytes);
}

bool ptr_aligned(const void* p, size_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Common checks of the pointer arrays.  Returns vSuccess and sets *aligned to the largest
// power-of-two alignment (up to 32 bytes) that every pointer has.
vResult_t check_ptrs(const vcomm* c, const void* const* send, void* const* recv, size_t esz,
                     int root, bool needAllSend, int* aligned, bool needAllRecv = true) {
    if (!send || !recv) return vInvalidArgument;
    uintptr_t bits = 32;
    for (int r = 0; r < c->nRanks; r++) {
        if (needAllSend || r == root) {
            if (!send[r] || !ptr_aligned(send[r], esz)) return vInvalidArgument;
            bits |= (uintptr_t)send[r];
        }
        if (needAllRecv || r == root) {
            if (!recv[r] || !ptr_aligned(recv[r], esz)) return vInvalidArgument;
            bits |= (uintptr_t)recv[r];
        }
    }
    *aligned = (int)(bits & (~bits + 1));       // lowest set bit, at most 32
    return vSuccess;
}

vResult_t make_plan(const vcomm* c, int coll, size_t count, int dt, int aligned, vPlanInfo_t* p) {
    vPlanRequest_t q;
    std::memset(&q, 0, sizeof(q));
    q.nRanks = c->nRanks;
    q.nChannels = c->nChannels;
    q.proto = c->proto;
    q.algo = c->cfg.algo;
    q.coll = coll;
    q.datatype = dt;
    q.count = count;
    q.chunkBytes = c->cfg.chunkBytes;
    q.aligned16 = aligned >= 16 ? 1 : 0;
    q.aligned32 = aligned >= 32 ? 1 : 0;
    q.noBulkCopy = c->cfg.bulkCopy ? 0 : 1;
    q.persistentGrid = c->cfg.persistentGrid ? 1 : 0;
    q.smCount = c->smCount;
    q.l2Bytes = c->l2Bytes;
    return vPlanCompute(&q, p);
}

bool stream_capturing(cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs != cudaStreamCaptureStatusNone;
}

// Record, on `stream`, the point after the launch just enqueued (one event per stream).
void track_launch(vcomm* c, cudaStream_t stream) {
    StreamEvent* slot = nullptr;
    for (auto& t : c->tracked)
        if (t.event && t.stream == stream) { slot = &t; break; }
    if (!slot) {
        for (auto& t : c->tracked)
            if (!t.event) { slot = &t; break; }
    }
    if (!slot) {                     // every slot in use: retire the oldest-assigned one
        slot = &c->tracked[c->trackedNext++ % kTrackedStreams];
        if (slot->recorded) cudaEventSynchronize(slot->event);
        slot->recorded = false;
    }
    if (!slot->event && cudaEventCreateWithFlags(&slot->event, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        cudaStreamSynchronize(stream);           // cannot track it: wait for it instead
        return;
    }
    slot->stream = stream;
    if (cudaEventRecord(slot->event, stream) == cudaSuccess) slot->recorded = true;
}

// Wait for every tracked launch (before freeing or replacing communicator memory).
void wait_tracked(vcomm* c) {
    for (auto& t : c->tracked)
        if (t.recorded) {
            cudaEventSynchronize(t.event);
            t.recorded = false;
        }
}

// usesComm: the kernel touches communicator memory (FIFOs, counters, the status word), so
// vcommDestroy must wait for it.  Launches that touch only the caller's buffers are not
// tracked: an event recorded between two kernels would also stop the second from being
// scheduled during the first one's tail (programmatic dependent launch).
vResult_t finish_launch(vcomm* c, cudaError_t e, cudaStream_t stream, const char* what, bool usesComm = false) {
    if (e != cudaSuccess) {
        c->hostError = vUnhandledCudaError;
        return cuda_fail(c, e, what);
    }
    // Eager launches only; launches captured into a graph run when the graph does, which
    // the caller orders.
    if (usesComm && !stream_capturing(stream)) track_launch(c, stream);
    return vSuccess;
}

void fill_onepass(vc::OnePassArgs* a, const vcomm* c, const void* const* send, void* const* recv,
                  const vPlanInfo_t& p, size_t count) {
    std::memset(a, 0, sizeof(*a));
    for (int r = 0; r < c->nRanks; r++) {
        a->send[r] = send ? send[r] : nullptr;
        a->recv[r] = recv[r];
    }
    a->orderRoot = -1;
    a->outRoot = -1;
    a->nRanks = c->nRanks;
    a->ctasPerChannel = p.ctasPerChannel;
    a->count = count;
    a->blockElems = p.blockElems;
    a->chanElems = p.channelElems;
    a->tileBytes = p.tileBytes ? p.tileBytes : (size_t)64 * 1024;
}

// Grow the ring FIFOs and control words if this plan needs more than the communicator has.
vResult_t ensure_fifo(vcomm* c, const vPlanInfo_t& p) {
    const size_t need = (size_t)c->nChannels * c->nRanks * p.fifoBytes;
    if (!c->ctrl) {
        const size_t ctrlBytes = (size_t)c->nChannels * c->nRanks * vc::kCtrlStride * sizeof(unsigned long long);
        cudaError_t e = cudaMalloc(&c->ctrl, ctrlBytes);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaMalloc(ctrl)");
        e = cudaMemset(c->ctrl, 0, ctrlBytes);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemset(ctrl)");
    }
    if (need <= c->fifoCap) return vSuccess;
    wait_tracked(c);                 // no launch may still use the FIFOs being replaced
    if (c->fifo) cudaFree(c->fifo);
    c->fifo = nullptr;
    c->fifoCap = 0;
    cudaError_t e = cudaMalloc(&c->fifo, need);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaMalloc(fifo)");
    e = cudaMemset(c->fifo, 0, need);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemset(fifo)");
    c->fifoCap = need;
    return vSuccess;
}

vResult_t launch_ring_plan(vcomm* c, int coll, const void* const* send, void* const* recv,
                           size_t count, vDataType_t dt, vRedOp_t op, vDataType_t outType, int root,
                           bool hasScale, float scale, const vPlanInfo_t& p, cudaStream_t stream) {
    if (!c->cooperative) return vInvalidUsage;
    int maxCtas = 0;
    cudaError_t e = vc::ring_max_coresident(dt, op, outType, (vProto_t)p.proto, p.threadsPerCta,
                                            c->smCount, &maxCtas);
    if (e != cudaSuccess) return cuda_fail(c, e, "occupancy");
    if (p.gridCtas > maxCtas) {
        if (c->cfg.debug)
            std::fprintf(stderr, "vcomm: ring needs %d co-resident CTAs, device holds %d\n", p.gridCtas, maxCtas);
        return vInvalidUsage;
    }
    const bool capturing = stream_capturing(stream);
    unsigned int epoch;
    if (capturing) {
        // A captured launch replays with the arguments it was captured with, so it cannot
        // carry a fresh epoch: the graph clears the control words before every replay and
        // uses epoch 1, which eager launches never use.  LL and LL128 keep their flags in
        // the FIFO lines, so for them the graph also clears the part of every slot that
        // this transfer can write (its largest per-channel step, in wire bytes); Simple
        // data is ordered by the counters alone.  FIFOs cannot be allocated during capture:
        // an eager ring call of at least this size must come first.
        const size_t need = (size_t)c->nChannels * c->nRanks * p.fifoBytes;
        if (!c->ctrl || need > c->fifoCap) return vInvalidUsage;
        const size_t ctrlBytes = (size_t)c->nChannels * c->nRanks * vc::kCtrlStride * sizeof(unsigned long long);
        e = cudaMemsetAsync(c->ctrl, 0, ctrlBytes, stream);
        if (e == cudaSuccess && p.proto != vProtoSimple) {
            const size_t esz = elem_size(dt);
            const size_t payload = std::min(p.slotPayloadElems, std::max<size_t>(1, p.channelElems)) * esz;
            size_t wire = p.proto == vProtoLL ? (payload + 7) / 8 * 16 : (payload + 119) / 120 * 128;
            wire = std::min(p.slotBytes, (wire + 127) / 128 * 128);
            e = cudaMemset2DAsync(c->fifo, p.slotBytes, 0, wire,
                                  (size_t)c->nChannels * c->nRanks * vc::kFifoSlots, stream);
        }
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemsetAsync(capture)");
        epoch = 1;
    } else {
        vResult_t res = ensure_fifo(c, p);
        if (res != vSuccess) return res;
        c->epoch++;
        if ((c->epoch & 0xFFu) <= 1u) {
            // LL flags keep only the low byte of the epoch: clear stale flags when it wraps.
            // Low bytes 0 (cleared memory) and 1 (captured graphs) are never used here.
            e = cudaMemsetAsync(c->fifo, 0, c->fifoCap, stream);
            if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemsetAsync(fifo)");
            c->epoch = (c->epoch & ~0xFFu) | 2u;
        }
        epoch = c->epoch;
    }
    vc::RingArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int r = 0; r < c->nRanks; r++) {
        a.send[r] = send[r];
        a.recv[r] = recv[r];
    }
    a.nRanks = c->nRanks;
    a.nChannels = c->nChannels;
    a.coll = coll;
    a.op = op;
    a.root = root;
    a.aligned = p.vectorized;
    a.hasScale = hasScale ? 1 : 0;
    a.scale = scale;
    switch (coll) {
    case vCollAllReduce: case vCollBroadcast: a.count = count; break;
    default: a.count = count * (size_t)c->nRanks; break;
    }
    a.blockElems = p.blockElems;
    a.chanElems = p.channelElems;
    a.chunkElems = p.chunkElems;
    a.slotElems = p.slotPayloadElems;
    a.slotBytes = p.slotBytes;
    a.fifo = c->fifo;
    a.ctrl = c->ctrl;
    a.epochHi = (unsigned long long)epoch << 32;
    a.llEpoch = (epoch & 0xFFu) << 24;
    a.timeoutNs = (unsigned long long)c->cfg.timeoutMs * 1000000ull;
    a.abortHost = c->abortHostDev;
    a.abortDev = c->abortDev;
    a.status = c->statusDev;
    a.statusHost = c->statusHostDev;
    a.testStallRank = c->testStallRank;
    a.testJitterNs = c->testJitterNs;
    a.testBadFlagRank = c->testBadFlagRank;
    e = vc::launch_ring(a, dt, op, outType, (vProto_t)p.proto, p.gridCtas, p.threadsPerCta, stream);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        return vInvalidUsage;
    }
    return finish_launch(c, e, stream, "ring launch", true);
}

// One launch for up to vc::group_capacity(N) recorded all-reduces of one type, op, stream
// and vector width.  The work table is built in the kernel's parameter block, which the
// launch copies, so the host copy is free for the next batch as soon as this returns.
vResult_t launch_group_batch(vcomm* c, const std::vector<const GroupRec*>& items) {
    const int N = c->nRanks;
    const GroupRec& r0 = *items[0];
    const size_t n = items.size();
    if (n > (size_t)vc::group_capacity(N)) return vInternalError;
    if (!c->groupArgs) {
        c->groupArgs = new (std::nothrow) vc::GroupArgs;
        if (!c->groupArgs) return vSystemError;
    }
    vc::GroupArgs& a = *c->groupArgs;
    const size_t itemBytes = (n * sizeof(vc::GroupItem) + 15) / 16 * 16;
    vc::GroupItem* it = reinterpret_cast<vc::GroupItem*>(a.table);
    const void** ptrs = reinterpret_cast<const void**>(a.table + itemBytes);
    const size_t esz = elem_size(r0.dt);
    const size_t U = r0.vecBytes ? (size_t)r0.vecBytes / esz : (size_t)vc::kElemsPerThread;
    unsigned long long units = 0;
    for (size_t i = 0; i < n; i++) {
        const GroupRec& g = *items[i];
        it[i].unitStart = units;
        it[i].count = g.count;
        it[i].blockElems = g.blockElems;
        it[i].unitsPerBlock = (g.blockElems + U - 1) / U;
        it[i].ptrOff = (int)(i * 2 * N);
        it[i].pad = 0;
        for (int r = 0; r < N; r++) {
            ptrs[i * 2 * N + r] = g.send[r];
            ptrs[i * 2 * N + N + r] = g.recv[r];
        }
        units += it[i].unitsPerBlock * (unsigned long long)N;
    }
    a.nItems = (int)n;
    a.nRanks = N;
    a.totalUnits = units;
    a.ptrByteOff = (int)itemBytes;
    a.pad = 0;
    // One thread per work unit, CTAs dispatched in order; one resident wave striding over
    // the units when the persistent grid is asked for or the work is under two waves.
    const unsigned long long need = (units + vc::kOnePassThreads - 1) / vc::kOnePassThreads;
    const unsigned long long resident = (unsigned long long)(r0.vecBytes == 32 ? 1 : 2) * c->smCount;
    const unsigned long long cap = (c->cfg.persistentGrid || need < 2 * resident) ? resident : vc::kMaxGridCtas;
    const int grid = (int)std::min<unsigned long long>(cap, std::max(1ull, need));
    const cudaError_t e = vc::launch_allreduce_group(a, r0.dt, r0.op, r0.vecBytes, grid, vc::kOnePassThreads,
                                                     r0.stream);
    return finish_launch(c, e, r0.stream, "group launch");
}

// Shared front half of every collective.
struct Front {
    vResult_t res;
    int aligned;        // common pointer alignment in bytes (up to 32)
};

Front front(vcomm* c, const void* const* send, void* const* recv, size_t count, int dt, int root,
            bool needAllSend, bool needAllRecv = true) {
    Front f{vSuccess, 0};
    if (!comm_ok(c)) { f.res = vInvalidArgument; return f; }
    vResult_t s = sticky(c);
    if (s != vSuccess) { f.res = s; return f; }
    const size_t esz = elem_size(dt);
    if (esz == 0) { f.res = vInvalidArgument; return f; }
    // N*N*count*esz must fit comfortably in size_t
    const size_t n2 = (size_t)c->nRanks * (size_t)c->nRanks;
    if (count > ((size_t)1 << 62) / (n2 * esz)) { f.res = vInvalidArgument; return f; }
    if (count == 0) return f;
    f.res = check_ptrs(c, send, recv, esz, root, needAllSend, &f.aligned, needAllRecv);
    return f;
}

bool valid_op(int op) { return op >= vSum && op <= vMax; }

std::vector<const void*> copy_ptrs(const void* const* p, int n) {
    return p ? std::vector<const void*>(p, p + n) : std::vector<const void*>(n, nullptr);
}
std::vector<void*> copy_ptrs(void* const* p, int n) {
    return p ? std::vector<void*>(p, p + n) : std::vector<void*>(n, nullptr);
}

// Inside a group every call is recorded (its pointer arrays copied) and runs at
// vcommGroupEnd.
#define VC_GROUP_RECORD(c, CALL)                                                           \
    do {                                                                                   \
        if ((c)->groupDepth > 0) {                                                         \
            GroupRec rec;                                                                  \
            rec.launch = CALL;                                                             \
            (c)->group->push_back(std::move(rec));                                         \
            return vSuccess;                                                               \
        }                                                                                  \
    } while (0)

}  // namespace

extern "C" {

const char* vcommGetErrorString(vResult_t r) {
    switch (r) {
    case vSuccess: return "no error";
    case vUnhandledCudaError: return "unhandled cuda error";
    case vSystemError: return "system error";
    case vInternalError: return "internal error";
    case vInvalidArgument: return "invalid argument";
    case vInvalidUsage: return "invalid usage";
    case vTimeout: return "timeout";
    case vInProgress: return "in progress";
    case vAborted: return "aborted";
    }
    return "unknown result code";
}

vResult_t vcommInit(vcomm_t* comm, int nRanks, int nChannels, vProto_t protocol) {
    if (!comm) return vInvalidArgument;
    *comm = nullptr;
    if (nRanks < 1 || nRanks > VCOMM_MAX_RANKS) return vInvalidArgument;
    if (nChannels < 1 || nChannels > VCOMM_MAX_CHANNELS) return vInvalidArgument;
    if (protocol < vProtoSimple || protocol > vProtoAuto) return vInvalidArgument;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
    vcomm* c = new (std::nothrow) vcomm();
    if (!c) return vSystemError;
    std::memset((void*)c, 0, sizeof(*c));
    c->cfg = Config();
    read_env(&c->cfg);
    c->nRanks = nRanks;
    c->nChannels = nChannels;
    c->proto = protocol;
    c->device = dev;
    c->testStallRank = -1;
    c->testBadFlagRank = -1;
    c->hostError = vSuccess;
    c->epoch = 1;                    // eager ring launches use epochs >= 2
    c->group = new (std::nothrow) std::vector<GroupRec>();
    if (!c->group) {
        free_comm(c);
        return vSystemError;
    }
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) goto fail;
    c->smCount = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) goto fail;
    c->l2Bytes = (size_t)v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) goto fail;
    c->cooperative = v;
    if ((e = cudaMalloc(&c->statusDev, sizeof(vc::Status))) != cudaSuccess) goto fail;
    if ((e = cudaMemset(c->statusDev, 0, sizeof(vc::Status))) != cudaSuccess) goto fail;
    if ((e = cudaMalloc(&c->abortDev, sizeof(unsigned int))) != cudaSuccess) goto fail;
    if ((e = cudaMemset(c->abortDev, 0, sizeof(unsigned int))) != cudaSuccess) goto fail;
    if ((e = cudaMalloc(&c->tileCounters, vc::kAllCounterSlots * 2 * sizeof(unsigned int))) != cudaSuccess)
        goto fail;
    if ((e = cudaMemset(c->tileCounters, 0, vc::kAllCounterSlots * 2 * sizeof(unsigned int))) != cudaSuccess)
        goto fail;
    if ((e = cudaHostAlloc(&c->statusHost, sizeof(vc::Status), cudaHostAllocMapped)) != cudaSuccess) goto fail;
    std::memset(c->statusHost, 0, sizeof(vc::Status));
    if ((e = cudaHostGetDevicePointer(&c->statusHostDev, c->statusHost, 0)) != cudaSuccess) goto fail;
    if ((e = cudaHostAlloc(&c->abortHost, sizeof(unsigned int), cudaHostAllocMapped)) != cudaSuccess) goto fail;
    *c->abortHost = 0;
    if ((e = cudaHostGetDevicePointer(&c->abortHostDev, c->abortHost, 0)) != cudaSuccess) goto fail;
    c->startMagic = c->endMagic = kMagic;
    *comm = c;
    return vSuccess;
fail:
    {
        vResult_t r = cuda_fail(c, e, "vcommInit");
        free_comm(c);
        return r;
    }
}

vResult_t vcommDestroy(vcomm_t c) {
    if (!comm_ok(c)) return vInvalidArgument;
    DeviceGuard g(c);
    wait_tracked(c);
    free_comm(c);
    return vSuccess;
}

vResult_t vcommCount(vcomm_t c, int* nRanks) {
    if (!comm_ok(c) || !nRanks) return vInvalidArgument;
    *nRanks = c->nRanks;
    return vSuccess;
}

vResult_t vcommGetAsyncError(vcomm_t c, vResult_t* err) {
    if (!comm_ok(c) || !err) return vInvalidArgument;
    *err = sticky(c);
    return vSuccess;
}

vResult_t vcommAbort(vcomm_t c) {
    if (!comm_ok(c)) return vInvalidArgument;
    *(volatile unsigned int*)c->abortHost = 1u;
    if (c->hostError == vSuccess) c->hostError = vAborted;
    return vSuccess;
}

vResult_t vcommGroupStart(vcomm_t c) {
    if (!comm_ok(c)) return vInvalidArgument;
    c->groupDepth++;
    return vSuccess;
}

vResult_t vcommGroupEnd(vcomm_t c) {
    NvtxRange nvtx_("vcommGroupEnd");
    if (!comm_ok(c)) return vInvalidArgument;
    if (c->groupDepth == 0) return vInvalidUsage;
    if (--c->groupDepth > 0) return vSuccess;
    std::vector<GroupRec> recs;
    recs.swap(*c->group);
    vResult_t s = sticky(c);
    if (s != vSuccess) return s;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vResult_t first = vSuccess;
    // Fused all-reduces: batches of one (type, op, stream, vector width), in order of
    // their first call; a batch of one runs on its own.
    std::vector<bool> done(recs.size(), false);
    for (size_t i = 0; i < recs.size(); i++) {
        if (!recs[i].fusable || done[i]) continue;
        std::vector<const GroupRec*> batch;
        for (size_t j = i; j < recs.size(); j++) {
            const GroupRec& a = recs[i];
            const GroupRec& b = recs[j];
            if (!b.fusable || done[j] || b.dt != a.dt || b.op != a.op || b.stream != a.stream ||
                b.vecBytes != a.vecBytes)
                continue;
            batch.push_back(&b);
            done[j] = true;
        }
        const bool single = batch.size() == 1;
        const size_t cap = (size_t)vc::group_capacity(c->nRanks);
        for (size_t k = 0; k < batch.size(); k += (single ? 1 : cap)) {
            vResult_t r;
            if (single) {
                const GroupRec& b = *batch[k];
                r = vAllReduce(b.send.data(), b.recv.data(), b.count, b.dt, b.op, c, b.stream);
            } else {
                std::vector<const GroupRec*> part(batch.begin() + k, batch.begin() + std::min(batch.size(), k + cap));
                r = launch_group_batch(c, part);
            }
            if (r != vSuccess && first == vSuccess) first = r;
        }
    }
    for (auto& rec : recs) {
        if (rec.fusable) continue;
        const vResult_t r = rec.launch();
        if (r != vSuccess && first == vSuccess) first = r;
    }
    return first;
}

vResult_t vcommSetAlgo(vcomm_t c, vAlgo_t algo) {
    if (!comm_ok(c) || algo < vAlgoAuto || algo > vAlgoTree) return vInvalidArgument;
    c->cfg.algo = algo;
    return vSuccess;
}

vResult_t vcommSetProtocol(vcomm_t c, vProto_t proto) {
    if (!comm_ok(c) || proto < vProtoSimple || proto > vProtoAuto) return vInvalidArgument;
    c->proto = proto;
    return vSuccess;
}

vResult_t vcommSetChunkBytes(vcomm_t c, size_t chunkBytes) {
    if (!comm_ok(c)) return vInvalidArgument;
    if (chunkBytes != 0 &&
        (chunkBytes < 4096 || chunkBytes > (64u << 20) || (chunkBytes & (chunkBytes - 1)) != 0))
        return vInvalidArgument;
    c->cfg.chunkBytes = chunkBytes;
    return vSuccess;
}

vResult_t vcommSetTimeoutMs(vcomm_t c, int timeoutMs) {
    if (!comm_ok(c) || timeoutMs < 1) return vInvalidArgument;
    c->cfg.timeoutMs = timeoutMs;
    return vSuccess;
}

vResult_t vcommTestSetStallRank(vcomm_t c, int rank) {
    if (!comm_ok(c) || rank < -1 || rank >= c->nRanks) return vInvalidArgument;
    c->testStallRank = rank;
    return vSuccess;
}

vResult_t vcommTestSetBadFlagRank(vcomm_t c, int rank) {
    if (!comm_ok(c) || rank < -1 || rank >= c->nRanks) return vInvalidArgument;
    c->testBadFlagRank = rank;
    return vSuccess;
}

vResult_t vcommTestSetJitterNs(vcomm_t c, unsigned int maxNs) {
    if (!comm_ok(c) || maxNs > 1000000u) return vInvalidArgument;
    c->testJitterNs = maxNs;
    return vSuccess;
}

vResult_t vcommQueryPlan(vcomm_t c, vColl_t coll, size_t count, vDataType_t dt, int aligned,
                         vPlanInfo_t* plan) {
    if (!comm_ok(c) || !plan) return vInvalidArgument;
    return make_plan(c, coll, count, dt, aligned, plan);
}

vResult_t vAllReduce(const void* const* send, void* const* recv, size_t count, vDataType_t dt,
                     vRedOp_t op, vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vAllReduce");
    Front f = front(c, send, recv, count, dt, 0, true);
    if (f.res != vSuccess || count == 0) return f.res;
    if (!valid_op(op)) return vInvalidArgument;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollAllReduce, count, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    if (c->groupDepth > 0) {
        GroupRec rec;
        rec.send = copy_ptrs(send, c->nRanks);
        rec.recv = copy_ptrs(recv, c->nRanks);
        rec.count = count;
        rec.dt = dt;
        rec.op = op;
        rec.stream = stream;
        rec.vecBytes = p.vecBytes;
        rec.blockElems = p.blockElems;
        rec.fusable = p.algo == vAlgoOnePass;
        if (!rec.fusable) {
            auto s_ = rec.send;
            auto r_ = rec.recv;
            rec.launch = [=]() { return vAllReduce(s_.data(), r_.data(), count, dt, op, c, stream); };
        }
        c->group->push_back(std::move(rec));
        return vSuccess;
    }
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    debug_plan(c, vCollAllReduce, count, dt, p);
    if (p.algo == vAlgoRing)
        return launch_ring_plan(c, vCollAllReduce, send, recv, count, dt, op, dt, 0, false, 1.0f, p, stream);
    if (p.algo == vAlgoTree) {
        vc::TreeArgs ta;
        std::memset(&ta, 0, sizeof(ta));
        for (int r = 0; r < c->nRanks; r++) {
            ta.send[r] = send[r];
            ta.recv[r] = recv[r];
        }
        ta.nRanks = c->nRanks;
        ta.count = count;
        ta.split = std::min(p.blockElems, count);
        for (int t = 0; t < 2; t++) {
            // post-order of tree t: children before parents, child 0's subtree first
            int root = 0;
            for (int v = 0; v < c->nRanks; v++) {
                int u, a0, a1;
                vPlanTreeLinks(c->nRanks, v, t, &u, &a0, &a1);
                if (u < 0) root = v;
            }
            int n = 0;
            std::function<void(int)> visit = [&](int v) {
                int u, a0, a1;
                vPlanTreeLinks(c->nRanks, v, t, &u, &a0, &a1);
                int kids = 0;
                if (a0 >= 0) { visit(a0); kids++; }
                if (a1 >= 0) { visit(a1); kids++; }
                ta.prog[t][n] = (signed char)v;
                ta.nchild[t][n] = (signed char)kids;
                n++;
            };
            visit(root);
        }
        return finish_launch(c, vc::launch_allreduce_tree(ta, dt, op, p.vecBytes, p.gridCtas, p.threadsPerCta,
                                                          stream), stream, "allreduce tree");
    }
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, count);
    return finish_launch(c, vc::launch_allreduce_onepass(a, dt, op, p.vecBytes, p.gridCtas,
                                                         p.threadsPerCta, stream), stream, "allreduce");
}

static vResult_t reduce_scatter_impl(const void* const* send, void* const* recv, size_t rc,
                                     vDataType_t dt, vRedOp_t op, vDataType_t outType, bool hasScale,
                                     float scale, vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vReduceScatter");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return reduce_scatter_impl(s_.data(), r_.data(), rc, dt, op, outType, hasScale, scale, c, stream); });
    }
    Front f = front(c, send, recv, rc, dt, 0, true);
    if (f.res != vSuccess || rc == 0) return f.res;
    if (!valid_op(op)) return vInvalidArgument;
    if (outType != dt && !(outType == vFloat32 && (dt == vFloat16 || dt == vBFloat16))) return vInvalidArgument;
    for (int r = 0; r < c->nRanks; r++)
        if (!ptr_aligned(recv[r], elem_size(outType))) return vInvalidArgument;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollReduceScatter, rc, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollReduceScatter, rc, dt, p);
    if (p.algo == vAlgoRing)
        return launch_ring_plan(c, vCollReduceScatter, send, recv, rc, dt, op, outType, 0, hasScale, scale, p,
                                stream);
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, rc * (size_t)c->nRanks);
    a.hasScale = hasScale ? 1 : 0;
    a.scale = scale;
    return finish_launch(c, vc::launch_reduce_scatter_onepass(a, dt, op, outType, p.vecBytes,
                                                              p.gridCtas, p.threadsPerCta, stream),
                         stream, "reduce_scatter");
}

vResult_t vReduceScatter(const void* const* send, void* const* recv, size_t recvcount, vDataType_t dt,
                         vRedOp_t op, vcomm_t c, cudaStream_t stream) {
    return reduce_scatter_impl(send, recv, recvcount, dt, op, dt, false, 1.0f, c, stream);
}

vResult_t vReduceScatterScaleCast(const void* const* send, void* const* recv, size_t recvcount,
                                  vDataType_t dt, vRedOp_t op, vDataType_t outType, float scale,
                                  vcomm_t c, cudaStream_t stream) {
    if (dt == vInt32) return vInvalidArgument;
    return reduce_scatter_impl(send, recv, recvcount, dt, op, outType, true, scale, c, stream);
}

vResult_t vAllGather(const void* const* send, void* const* recv, size_t sendcount, vDataType_t dt,
                     vRedOp_t op, vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vAllGather");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vAllGather(s_.data(), r_.data(), sendcount, dt, op, c, stream); });
    }
    (void)op;
    Front f = front(c, send, recv, sendcount, dt, 0, true);
    if (f.res != vSuccess || sendcount == 0) return f.res;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollAllGather, sendcount, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollAllGather, sendcount, dt, p);
    if (p.algo == vAlgoRing)
        return launch_ring_plan(c, vCollAllGather, send, recv, sendcount, dt, vSum, dt, 0, false, 1.0f, p, stream);
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, sendcount);
    if (p.bulkCopy)
        return finish_launch(c, vc::launch_fanout_tma(a, (int)elem_size(dt), false, p.gridCtas, p.tmaStages, c->statusDev,
                                                      c->statusHostDev, stream), stream, "allgather", true);
    return finish_launch(c, vc::launch_allgather_onepass(a, (int)elem_size(dt), p.vecBytes, p.gridCtas,
                                                         p.threadsPerCta, stream), stream, "allgather");
}

vResult_t vBroadcast(const void* const* send, void* const* recv, size_t count, vDataType_t dt,
                     vRedOp_t op, int root, vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vBroadcast");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vBroadcast(s_.data(), r_.data(), count, dt, op, root, c, stream); });
    }
    (void)op;
    if (!comm_ok(c)) return vInvalidArgument;
    if (root < 0 || root >= c->nRanks) return vInvalidArgument;
    Front f = front(c, send, recv, count, dt, root, false);
    if (f.res != vSuccess || count == 0) return f.res;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollBroadcast, count, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollBroadcast, count, dt, p);
    if (p.algo == vAlgoRing) {
        const void* sends[VCOMM_MAX_RANKS];
        for (int i = 0; i < c->nRanks; i++) sends[i] = send[i];
        return launch_ring_plan(c, vCollBroadcast, sends, recv, count, dt, vSum, dt, root, false, 1.0f, p, stream);
    }
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, count);
    a.root = root;
    if (p.bulkCopy)
        return finish_launch(c, vc::launch_fanout_tma(a, (int)elem_size(dt), true, p.gridCtas, p.tmaStages, c->statusDev,
                                                      c->statusHostDev, stream), stream, "broadcast", true);
    return finish_launch(c, vc::launch_broadcast_onepass(a, (int)elem_size(dt), p.vecBytes, p.gridCtas,
                                                         p.threadsPerCta, stream), stream, "broadcast");
}

vResult_t vAllToAll(const void* const* send, void* const* recv, size_t count, vDataType_t dt,
                    vRedOp_t op, vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vAllToAll");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vAllToAll(s_.data(), r_.data(), count, dt, op, c, stream); });
    }
    (void)op;
    Front f = front(c, send, recv, count, dt, 0, true);
    if (f.res != vSuccess || count == 0) return f.res;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollAllToAll, count, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollAllToAll, count, dt, p);
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, count);
    return finish_launch(c, vc::launch_alltoall_onepass(a, (int)elem_size(dt), p.vecBytes, p.gridCtas,
                                                        p.threadsPerCta, stream), stream, "alltoall");
}

vResult_t vReduce(const void* const* send, void* const* recv, size_t count, vDataType_t dt, vRedOp_t op,
                  int root, vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vReduce");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vReduce(s_.data(), r_.data(), count, dt, op, root, c, stream); });
    }
    if (!comm_ok(c)) return vInvalidArgument;
    if (root < 0 || root >= c->nRanks || !valid_op(op)) return vInvalidArgument;
    Front f = front(c, send, recv, count, dt, root, true, false);
    if (f.res != vSuccess || count == 0) return f.res;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollReduce, count, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollReduce, count, dt, p);
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, count);
    a.orderRoot = root;
    a.outRoot = root;
    return finish_launch(c, vc::launch_allreduce_onepass(a, dt, op, p.vecBytes, p.gridCtas, p.threadsPerCta,
                                                         stream), stream, "reduce");
}

vResult_t vGather(const void* const* send, void* const* recv, size_t sendcount, vDataType_t dt, int root,
                  vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vGather");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vGather(s_.data(), r_.data(), sendcount, dt, root, c, stream); });
    }
    if (!comm_ok(c)) return vInvalidArgument;
    if (root < 0 || root >= c->nRanks) return vInvalidArgument;
    Front f = front(c, send, recv, sendcount, dt, root, true, false);
    if (f.res != vSuccess || sendcount == 0) return f.res;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollGather, sendcount, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollGather, sendcount, dt, p);
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, sendcount);
    a.outRoot = root;
    if (p.bulkCopy)
        return finish_launch(c, vc::launch_fanout_tma(a, (int)elem_size(dt), false, p.gridCtas, p.tmaStages, c->statusDev,
                                                      c->statusHostDev, stream), stream, "gather", true);
    return finish_launch(c, vc::launch_allgather_onepass(a, (int)elem_size(dt), p.vecBytes, p.gridCtas,
                                                         p.threadsPerCta, stream), stream, "gather");
}

vResult_t vScatter(const void* const* send, void* const* recv, size_t recvcount, vDataType_t dt, int root,
                   vcomm_t c, cudaStream_t stream) {
    NvtxRange nvtx_("vScatter");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vScatter(s_.data(), r_.data(), recvcount, dt, root, c, stream); });
    }
    if (!comm_ok(c)) return vInvalidArgument;
    if (root < 0 || root >= c->nRanks) return vInvalidArgument;
    Front f = front(c, send, recv, recvcount, dt, root, false, true);
    if (f.res != vSuccess || recvcount == 0) return f.res;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    vResult_t r = make_plan(c, vCollScatter, recvcount, dt, f.aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollScatter, recvcount, dt, p);
    vc::OnePassArgs a;
    fill_onepass(&a, c, send, recv, p, recvcount);
    a.root = root;
    return finish_launch(c, vc::launch_scatter_onepass(a, (int)elem_size(dt), p.vecBytes, p.gridCtas,
                                                       p.threadsPerCta, stream), stream, "scatter");
}

vResult_t vAllToAllv(const void* const* send, void* const* recv, const int32_t* counts,
                     const int32_t* sdispls, const int32_t* rdispls, vDataType_t dt, vcomm_t c,
                     cudaStream_t stream) {
    NvtxRange nvtx_("vAllToAllv");
    if (comm_ok(c) && c->groupDepth > 0) {
        auto s_ = copy_ptrs(send, c->nRanks);
        auto r_ = copy_ptrs(recv, c->nRanks);
        VC_GROUP_RECORD(c, [=]() { return vAllToAllv(s_.data(), r_.data(), counts, sdispls, rdispls, dt, c, stream); });
    }
    if (!comm_ok(c)) return vInvalidArgument;
    vResult_t s = sticky(c);
    if (s != vSuccess) return s;
    const size_t esz = elem_size(dt);
    if (esz == 0 || !counts || !sdispls || !rdispls || !send || !recv) return vInvalidArgument;
    // NULL entries are allowed (a rank with nothing to send or receive); the kernel
    // rejects a positive count that would touch one.
    uintptr_t bits = 32;
    for (int i = 0; i < c->nRanks; i++) {
        if ((send[i] && !ptr_aligned(send[i], esz)) || (recv[i] && !ptr_aligned(recv[i], esz)))
            return vInvalidArgument;
        bits |= (uintptr_t)send[i] | (uintptr_t)recv[i];
    }
    const int aligned = (int)(bits & (~bits + 1));
    vResult_t r;
    DeviceGuard g(c);
    if (!g.ok) return vUnhandledCudaError;
    vPlanInfo_t p;
    r = make_plan(c, vCollAllToAllv, 0, dt, aligned, &p);
    if (r != vSuccess) return r;
    debug_plan(c, vCollAllToAllv, 0, dt, p);
    vc::A2AvArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int i = 0; i < c->nRanks; i++) {
        a.send[i] = send[i];
        a.recv[i] = recv[i];
    }
    a.counts = counts;
    a.sdispls = sdispls;
    a.rdispls = rdispls;
    a.nRanks = c->nRanks;
    a.elemSize = (int)esz;
    a.tileBytes = 64 * 1024;
    // A captured launch replays with the pair it was captured with: it takes one of the
    // captured set, which eager launches never rotate into.
    const size_t pair = stream_capturing(stream)
                            ? vc::kTileCounterSlots + (size_t)(c->capturedCounterSeq++ % vc::kCapturedCounterSlots)
                            : (size_t)(c->tileCounterSeq++ % vc::kTileCounterSlots);
    a.tileCounter = c->tileCounters + 2 * pair;
    a.status = c->statusDev;
    a.statusHost = c->statusHostDev;
    return finish_launch(c, vc::launch_alltoallv(a, p.gridCtas, p.threadsPerCta, stream), stream, "alltoallv",
                         true);
}

}  // extern "C"
