// planner.cpp -- host-side planning of one collective: block partition, channel split,
// ring chunk/slot geometry, algorithm and protocol choice, launch shape.  Pure host
// arithmetic with no CUDA calls, so it is unit-tested without a GPU.
//
// Sources for the rules:
//  * block size B = alignUp(ceil(count / N), 16 / elemSize): the tail-chunk rule of
//    RingARAlgorithm::getNextSendAddr (NCCL book section 2.3);
//  * channels: each channel owns count / nChannels of the data (NCCL book section 2.2,
//    channel walkthrough step 3); here the split is applied inside every block, rounded
//    up to 16 bytes, so a channel's share of each block starts on a vector boundary;
//  * ring geometry: FIFOs of NCCL_STEPS = 8 slots, a chunk = ALLREDUCE_CHUNKSTEPS = 4
//    slots, a slice = ALLREDUCE_SLICESTEPS = 2 slots (NCCL book chapter 6, ncclInfo);
//  * protocol payload: LL carries half the bytes of its slots, LL128 120 of every 128
//    (NCCL book chapter 5, ring.cc: busBw * 0.5 for LL, * 0.92 = 120/128 for LL128);
//  * bus bandwidth factor nSteps / nRanks with nSteps = 2(N-1) for all-reduce and N-1
//    otherwise (NCCL book chapter 5, ring.cc, algBw = busBw * nRanks / nSteps).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "internal.h"

namespace {

size_t elem_size(int dt) {
    switch (dt) {
    case vFloat32: case vInt32: return 4;
    case vFloat16: case vBFloat16: return 2;
    default: return 0;
    }
}

size_t div_up(size_t a, size_t b) { return (a + b - 1) / b; }
size_t align_up(size_t a, size_t b) { return div_up(a, b) * b; }

size_t pow2_floor(size_t x) {
    size_t p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

// ---- cost model ---------------------------------------------------------------------------
//
// The ring model of the NCCL book chapter 5 (ring.cc): time = latency + bus bytes / bus
// bandwidth, where a collective of S bytes per rank moves S * nSteps / N bus bytes
// (nSteps = 2(N-1) for all-reduce, N-1 otherwise), and LL / LL128 trade bandwidth for
// latency.  Fitted on GB300 per collective and protocol at 1, 8 and 32 channels
// (collective_communication_virtual_gb300/calibrate.py, from the staged-ring times in
// ring_timings_gb300.json: fp32 sum over 8 ranks, default chunks, 1 KiB .. 1 GiB per rank)
// with one more term each, which the data ask for:
//  * ring steps (all-reduce, reduce-scatter, all-gather):
//    lat + f min(x, knee) + max(0, x - knee) / rate -- below the knee a transfer is one
//    slot per step and its bytes cost f each, in turn at every step; above it the slots
//    pipeline and a byte costs 1 / rate;
//  * broadcast (a chain): lat + c sqrt(x) + x / rate -- the pipeline fill of a chain whose
//    slot count grows as sqrt(x) (the broadcast slot rule below).
// x is bytes per rank at 8 ranks; for N ranks the latency scales by nSteps, the ring
// steps' bytes by the bus bytes per rank byte (nSteps / N) and the chain's fill by
// sqrt(N - 2).  Channel counts between the anchors interpolate in log2; beyond 32 the fit
// is held flat.  The one-pass kernels are modelled as latency + minimum HBM bytes / rate.
struct RingFit {
    double latUs[3];           // at 1, 8, 32 channels
    double bytesPerUs[3];      // bytes per rank per microsecond, at 8 ranks
    double shape[3];           // ring steps: knee (bytes per rank); broadcast: sqrt coefficient
    double usPerMiBBelow[3];   // ring steps: microseconds per MiB below the knee
};
const RingFit kRingFit[4][3] = {                         // calibrate.py prints these
    {  // allreduce
        {{32.78, 34.64, 36.88}, {8645.7, 67998.5, 136493.1}, {524288, 262144, 67108864}, {94.19, 38.18, 5.87}},   // simple
        {{25.10, 23.29, 23.91}, {4334.9, 27992.4, 76631.0}, {524288, 524288, 2097152}, {145.06, 17.36, 9.21}},   // ll
        {{52.89, 50.81, 52.55}, {8766.1, 65218.3, 134180.0}, {2097152, 16777216, 67108864}, {85.25, 13.40, 6.00}},   // ll128
    },
    {  // reduce_scatter
        {{19.07, 20.07, 19.78}, {12499.0, 97454.3, 240898.1}, {4194304, 4194304, 67108864}, {50.13, 6.81, 3.34}},   // simple
        {{15.20, 13.40, 13.82}, {6096.0, 45305.2, 136545.6}, {2097152, 131072, 16777216}, {98.03, 0.00, 7.34}},   // ll
        {{31.41, 28.93, 28.64}, {15038.4, 115527.7, 312633.3}, {2097152, 16777216, 2097152}, {44.38, 7.69, 9.43}},   // ll128
    },
    {  // allgather
        {{18.31, 18.34, 18.25}, {23649.7, 171135.6, 288958.2}, {524288, 8388608, 67108864}, {33.08, 5.15, 2.80}},   // simple
        {{16.24, 12.94, 14.08}, {12006.0, 61903.8, 162660.8}, {65536, 16777216, 262144}, {32.94, 14.07, 1.37}},   // ll
        {{27.45, 25.14, 26.20}, {18657.9, 134711.5, 256851.9}, {4194304, 16777216, 67108864}, {46.17, 6.69, 3.35}},   // ll128
    },
    {  // broadcast
        {{15.26, 14.93, 15.57}, {23417.9, 177952.6, 353129.7}, {0.04029, 0.01383, 0.00713}, {0.00, 0.00, 0.00}},   // simple
        {{10.51, 7.78, 8.03}, {10609.6, 64002.3, 116232.2}, {0.00000, 0.00566, 0.00711}, {0.00, 0.00, 0.00}},   // ll
        {{19.99, 19.25, 19.89}, {19703.6, 159264.7, 368990.6}, {0.04487, 0.01849, 0.01648}, {0.00, 0.00, 0.00}},   // ll128
    },
};
// median relative error 0.022, max 0.241 over 396 points
const double kOnePassLatUs = 1.5;
const double kOnePassBytesPerUs = 7.097e6;                   // minimum bytes / (time - latency)

double interp_ch(const double v[3], int ch) {
    const double x = ch <= 1 ? 0.0 : (ch >= 32 ? 5.0 : std::log2((double)ch));
    if (x <= 3.0) return v[0] + (v[1] - v[0]) * (x / 3.0);
    return v[1] + (v[2] - v[1]) * ((x - 3.0) / 2.0);
}

int n_steps(int coll, int N) { return coll == vCollAllReduce ? 2 * (N - 1) : N - 1; }

int fit_row(int coll) {
    switch (coll) {
    case vCollAllReduce: return 0;
    case vCollReduceScatter: return 1;
    case vCollAllGather: return 2;
    default: return 3;
    }
}

double predict_ring_us(int proto, int coll, int N, int nCh, double bytesPerRank) {
    const RingFit& f = kRingFit[fit_row(coll)][proto];
    const double lat = interp_ch(f.latUs, nCh) * n_steps(coll, N) / n_steps(coll, 8);
    const double rate = interp_ch(f.bytesPerUs, nCh), shape = interp_ch(f.shape, nCh);
    if (coll == vCollBroadcast)
        return lat + shape * std::sqrt(bytesPerRank * std::max(0, N - 2) / 6.0) + bytesPerRank / rate;
    const double scale = ((double)n_steps(coll, N) / N) / ((double)n_steps(coll, 8) / 8.0);
    const double x = bytesPerRank * scale, below = interp_ch(f.usPerMiBBelow, nCh) / (1 << 20);
    return lat + below * std::min(x, shape) + std::max(0.0, x - shape) / rate;
}

double predict_onepass_us(double minBytes) { return kOnePassLatUs + minBytes / kOnePassBytesPerUs; }

}  // namespace

extern "C" vResult_t vPlanCompute(const vPlanRequest_t* q, vPlanInfo_t* p) {
    if (!q || !p) return vInvalidArgument;
    std::memset(p, 0, sizeof(*p));
    const int N = q->nRanks;
    if (N < 1 || N > VCOMM_MAX_RANKS) return vInvalidArgument;
    if (q->nChannels < 1 || q->nChannels > VCOMM_MAX_CHANNELS) return vInvalidArgument;
    if (q->coll < vCollAllReduce || q->coll > vCollScatter) return vInvalidArgument;
    if (q->proto < vProtoSimple || q->proto > vProtoAuto) return vInvalidArgument;
    if (q->algo < vAlgoAuto || q->algo > vAlgoTree) return vInvalidArgument;
    const size_t esz = elem_size(q->datatype);
    if (esz == 0) return vInvalidArgument;
    if (q->chunkBytes != 0 && (q->chunkBytes < 4096 || q->chunkBytes > (64u << 20) ||
                               (q->chunkBytes & (q->chunkBytes - 1)) != 0))
        return vInvalidArgument;
    const size_t VE = 16 / esz;
    const size_t count = q->count;
    const int smCount = q->smCount > 0 ? q->smCount : 152;

    // ---- blocks -----------------------------------------------------------------------
    size_t B = 0;          // elements per rank block
    size_t total = 0;      // elements of the block space (what channel ranges clamp to)
    switch (q->coll) {
    case vCollAllReduce: B = align_up(div_up(count, (size_t)N), VE); total = count; break;
    case vCollReduceScatter: B = count; total = count * (size_t)N; break;
    case vCollAllGather: B = count; total = count * (size_t)N; break;
    case vCollBroadcast: B = count; total = count; break;
    case vCollAllToAll: B = count; total = count * (size_t)N * (size_t)N; break;
    case vCollAllToAllv: B = 0; total = 0; break;
    case vCollReduce: B = align_up(div_up(count, (size_t)N), VE); total = count; break;
    case vCollGather: B = count; total = count * (size_t)N; break;
    case vCollScatter: B = count; total = count * (size_t)N; break;
    }
    p->blockElems = B;
    p->nChannels = q->nChannels;
    // Channel ranges start on 32 bytes, so either vector width fits inside them.
    p->channelElems = B ? align_up(div_up(B, (size_t)q->nChannels), 32 / esz) : 0;

    // ---- vector path ------------------------------------------------------------------
    bool vec = q->aligned16 != 0;
    if (q->coll == vCollReduceScatter || q->coll == vCollAllGather || q->coll == vCollAllToAll ||
        q->coll == vCollGather || q->coll == vCollScatter)
        vec = vec && (count % VE == 0);        // block starts r*count must stay 16-byte aligned
    p->vectorized = vec ? 1 : 0;
    // 32-byte accesses when every block (and so every vector) starts on 32 bytes.
    const bool v32 = vec && q->aligned32 != 0 && (B * esz) % 32 == 0;
    p->vecBytes = v32 ? 32 : vec ? 16 : 0;

    // ---- traffic model ----------------------------------------------------------------
    const double S = (double)count * (double)esz;
    switch (q->coll) {
    case vCollAllReduce: p->minBytes = 2.0 * N * S; p->busFactor = 2.0 * (N - 1) / N; break;
    case vCollReduceScatter: p->minBytes = (double)N * N * S + N * S; p->busFactor = (double)(N - 1) / N; break;
    case vCollAllGather: p->minBytes = (double)N * S + (double)N * N * S; p->busFactor = (double)(N - 1) / N; break;
    case vCollBroadcast: p->minBytes = S + (double)N * S; p->busFactor = (double)(N - 1) / N; break;
    case vCollAllToAll: p->minBytes = 2.0 * N * N * S; p->busFactor = (double)(N - 1) / N; break;
    case vCollReduce: p->minBytes = (double)N * S + S; p->busFactor = (double)(N - 1) / N; break;
    case vCollGather: case vCollScatter: p->minBytes = 2.0 * N * S; p->busFactor = (double)(N - 1) / N; break;
    default: p->minBytes = 0; p->busFactor = (double)(N - 1) / N; break;
    }

    // ---- algorithm and protocol: fixed by the caller, or the cheaper predicted time ----
    const bool ringable = N > 1 && (q->coll == vCollAllReduce || q->coll == vCollReduceScatter ||
                                    q->coll == vCollAllGather || q->coll == vCollBroadcast);
    const double bytesPerRank = q->coll == vCollAllGather ? S * N : q->coll == vCollReduceScatter ? S * N : S;
    int ringProto = q->proto;
    if (ringProto == vProtoAuto) {
        double best = 0;
        for (int pr = vProtoSimple; pr <= vProtoLL128; pr++) {
            const double t = predict_ring_us(pr, q->coll, N, q->nChannels, bytesPerRank);
            if (pr == vProtoSimple || t < best) { best = t; ringProto = pr; }
        }
    }
    const double tOne = predict_onepass_us(p->minBytes);
    const double tRing = ringable ? predict_ring_us(ringProto, q->coll, N, q->nChannels, bytesPerRank) : 0.0;
    bool ring = ringable && (q->algo == vAlgoRing || (q->algo == vAlgoAuto && tRing < tOne));
    p->algo = ring ? vAlgoRing : vAlgoOnePass;
    if (q->algo == vAlgoTree && q->coll == vCollAllReduce && N > 1) {
        // Double binary tree, one pass: two "blocks", the halves of the buffer.
        p->algo = vAlgoTree;
        p->blockElems = align_up(div_up(count, (size_t)2), VE);
        if (p->vecBytes == 32 && (p->blockElems * esz) % 32 != 0) p->vecBytes = 16;
        p->proto = q->proto == vProtoAuto ? vProtoSimple : q->proto;
        p->nChannels = 1;
        p->threadsPerCta = vc::kOnePassThreads;
        const size_t unit = p->vecBytes ? p->vecBytes / esz : 1;
        const size_t work = div_up(count, unit);
        // The 8-rank 32-byte kernel keeps its vectors in registers (one CTA per SM); the
        // others fit two per SM.
        const size_t resident = (size_t)((N == 8 && p->vecBytes == 32) ? 1 : 2) * smCount;
        if (!q->persistentGrid)                       // small work: smaller CTAs, more SMs
            while (p->threadsPerCta > 64 && div_up(work, (size_t)p->threadsPerCta) < (size_t)smCount)
                p->threadsPerCta /= 2;
        const size_t need = div_up(work, (size_t)p->threadsPerCta);
        const size_t cap = (q->persistentGrid || need < 2 * resident) ? resident : (size_t)vc::kMaxGridCtas;
        p->ctasPerChannel = (int)std::max<size_t>(1, std::min<size_t>(cap, need));
        p->gridCtas = p->ctasPerChannel;
        p->predictedUs = tOne;
        p->launches = 1;
        return vSuccess;
    }
    p->predictedUs = ring ? tRing : (q->coll == vCollAllToAllv ? 0.0 : tOne);
    p->launches = 1;

    if (!ring) {
        // One pass.  Default ("flat"): one CTA per slice of work -- a 512-thread CTA per
        // 512 vectors of every rank for the reductions, per 16-64 KiB tile for the copies
        // -- so the hardware hands CTAs out in order and the DRAM pages in use at any moment
        // stay within a narrow window of every buffer.  A persistent grid of one resident
        // wave whose CTAs stride over the work lets the CTAs drift apart and spreads the
        // accesses; measured on GB300 (8 ranks x 64 MiB fp32) it is 8-10 % slower.  It
        // stays selectable (persistentGrid) for comparison.
        p->proto = q->proto == vProtoAuto ? vProtoSimple : q->proto;
        // Reductions: smaller CTAs fit more threads on an SM beside a kernel's registers
        // (the 8-rank 32-byte reduce-scatter keeps 84: one 512-thread CTA per SM, but six of
        // 128 threads).  Measured on GB300, 128-thread CTAs take the 8-rank FSDP bucket's
        // reduce-scatter from 0.93 to 0.99 of the copy bandwidth, and 256-thread CTAs gain
        // 1-2 % for all-reduce below 64 MiB per rank.  The persistent shape keeps 512.
        p->threadsPerCta = vc::kOnePassThreads;
        if (!q->persistentGrid) {
            if (q->coll == vCollReduceScatter) p->threadsPerCta = 128;
            else if (q->coll == vCollAllReduce || q->coll == vCollReduce) p->threadsPerCta = 256;
        }
        // One resident wave (the persistent shape, and the cap for small work): rounded down
        // so it never spills into a second, mostly idle wave.  The 32-byte reduction kernels
        // hold up to 128 registers, 512 threads per SM; the copies fit twice that.
        const bool wide = p->vecBytes == 32 && (q->coll == vCollAllReduce || q->coll == vCollReduceScatter ||
                                                q->coll == vCollReduce);
        const int target = (wide ? 1 : 2) * smCount * (vc::kOnePassThreads / p->threadsPerCta);
        int per = std::max(1, target / q->nChannels);
        // Never more CTAs than a channel has work items: for the reductions a work item is
        // one thread's unit (a vector of every rank), for the copies a tile.
        size_t maxPer = 1;
        if (q->coll == vCollAllToAllv) {
            maxPer = (size_t)target;
        } else {
            const size_t chElems = std::min(p->channelElems, B);
            if (q->coll == vCollAllReduce || q->coll == vCollReduceScatter || q->coll == vCollReduce) {
                // a thread's unit: one vector of every rank, or on the element path 8
                // elements of every rank (32 of a warp's lanes times 8 per warp tile)
                // (the reduce-scatter element path of 2 to 4 ranks takes 4 16-byte vectors per
                // thread, of 8 ranks and 2-byte elements 1)
                const bool tiled = !p->vecBytes && q->coll == vCollReduceScatter &&
                                   ((N >= 2 && N <= 4) || (N == 8 && esz == 2));
                const size_t unit = p->vecBytes ? p->vecBytes / esz
                                                : tiled ? (16 / esz) * (N == 8 ? 1 : 4) : (size_t)vc::kElemsPerThread;
                const size_t units = div_up(chElems, unit) * (size_t)N;
                // Small work: smaller CTAs (down to 64 threads) spread it over more SMs
                // instead of loading a few SMs with 512 threads each.
                if (!q->persistentGrid)
                    while (p->threadsPerCta > 64 &&
                           div_up(units * (size_t)q->nChannels, (size_t)p->threadsPerCta) < (size_t)smCount)
                        p->threadsPerCta /= 2;
                maxPer = div_up(units, (size_t)p->threadsPerCta);
            } else {
                size_t blocks = q->coll == vCollBroadcast ? 1 : q->coll == vCollAllToAll ? (size_t)N * N : (size_t)N;
                // Copies: 64 KiB tiles (128 bytes in flight per thread of a 512-thread CTA)
                // unless that leaves fewer than 8 tiles per SM; then 32 or 16 KiB tiles, so the
                // last, partly filled wave is a smaller share of the launch.  The fan-out
                // copies (all-gather, broadcast: 8 stores per loaded byte) go on halving to
                // 8 KiB while there are fewer than 16 tiles per SM: measured on GB300, the
                // 8-rank FSDP bucket all-gather (3.125 MiB bf16 per rank) takes 37.5 us with
                // 16 KiB tiles and 36.5 us with 8 KiB (4 KiB: 37.3).
                // Small messages: tiles down to 2 KiB until there is a tile for every SM.
                const bool fanoutCopy = q->coll == vCollAllGather || q->coll == vCollBroadcast;
                size_t tile = (size_t)64 * 1024;
                auto tiles = [&](size_t t) { return div_up(chElems * esz, t) * blocks * (size_t)q->nChannels; };
                // Copies that 16-byte vectors cannot cover (ragged blocks, pointers off 16
                // bytes) take 32 KiB tiles: half the 64 KiB of a large vector copy (twice the
                // CTAs for loops that keep fewer bytes in flight per thread), twice the 16 KiB
                // the fan-out rule gives 2-byte all-gathers (half as many element heads,
                // tails and realignment set-ups per byte).  Measured on GB300 at
                // 64 MiB per rank with ragged blocks: bf16 all-gather 0.64 -> 0.77 (3 ranks)
                // and 0.76 -> 0.85 (8 ranks), fp32 all-to-all 0.88 -> 0.97 and 0.93 -> 1.01;
                // the fp32 all-gather (8 ranks) fell from 0.94 to 0.88, so 4-byte fan-out
                // copies keep the vector rule.
                if (!q->persistentGrid) {
                    if (vec || (fanoutCopy && esz == 4)) {
                        while (tile > 16 * 1024 && tiles(tile) < (size_t)8 * smCount) tile /= 2;
                        while (fanoutCopy && tile > 8 * 1024 && tiles(tile) < (size_t)16 * smCount) tile /= 2;
                    } else {
                        tile = (size_t)32 * 1024;
                    }
                    while (tile > 2 * 1024 && tiles(tile) < (size_t)smCount) tile /= 2;
                }
                p->tileBytes = tile;
                // A thread's share of a tile: 32 bytes where every loaded byte is stored to
                // all N ranks (all-gather, broadcast), 128 bytes where it is stored once
                // (all-to-all, gather, scatter), so a thread's loads and stores come to
                // about 256 bytes either way at 8 ranks; CTAs of 64 to 512 threads.
                // Measured on GB300 with 32 bytes for all: gather and scatter of 64 MiB at
                // the root ran at 0.87-0.89 of the copy bandwidth, against 0.98-1.03 with
                // 128, and the 8 x 4 MiB all-to-all took 14.1 us, against 7.2.
                const size_t perThread = fanoutCopy ? 32 : 128;
                p->threadsPerCta = (int)std::min<size_t>(vc::kOnePassThreads, std::max<size_t>(64, tile / perThread));
                maxPer = div_up(chElems * esz, tile) * blocks;
            }
        }
        maxPer = std::max<size_t>(1, maxPer);
        // Work of under two waves runs as one wave (a partly filled second wave costs
        // more than the drift of CTAs that stride at most twice).
        if (q->persistentGrid || q->coll == vCollAllToAllv || maxPer < 2 * (size_t)per)
            per = (int)std::min<size_t>((size_t)per, maxPer);
        else
            per = (int)std::min<size_t>((size_t)vc::kMaxGridCtas / (size_t)q->nChannels, maxPer);
        // Fan-out copies (all-gather, gather, broadcast) through TMA bulk copies: 16 KiB
        // tiles through shared memory, single-warp CTAs.
        const bool fanout = q->coll == vCollAllGather || q->coll == vCollGather || q->coll == vCollBroadcast;
        if (fanout && vec && q->noBulkCopy == 0 && (B * esz) % 16 == 0 && q->nChannels >= 1) {
            const size_t blocks = q->coll == vCollBroadcast ? 1 : (size_t)N;
            const size_t tiles = div_up(B * esz, (size_t)16 * 1024) * blocks;
            p->bulkCopy = 1;
            p->nChannels = 1;
            // Flat: one 16 KiB tile per single-stage CTA (about 13 resident per SM), handed
            // out in order.  Persistent: three 4-stage CTAs per SM striding over the tiles.
            p->tmaStages = q->persistentGrid ? 4 : 1;
            p->ctasPerChannel = q->persistentGrid ? (int)std::min<size_t>((size_t)vc::kTmaCtasPerSm * smCount, tiles)
                                                  : (int)std::min<size_t>((size_t)vc::kMaxGridCtas, tiles);
            p->gridCtas = p->ctasPerChannel;
            p->threadsPerCta = 32;
            return vSuccess;
        }
        if (q->coll == vCollAllToAllv) { p->nChannels = 1; per = smCount; }   // 1 CTA per SM
        p->ctasPerChannel = per;
        p->gridCtas = per * p->nChannels;
        (void)total;
        return vSuccess;
    }

    // ---- ring geometry ------------------------------------------------------------------
    // A chunk is chunkBytes of data per rank, 4 slots of chunkBytes / 4 data bytes each; a
    // slot's size in the FIFO follows the protocol: the same for Simple, twice for LL (a
    // flag beside every 4 data bytes), and whole 128-byte lines of 120 data bytes for LL128
    // (an even number of lines, so every slot starts on 256 bytes).  Sizing slots by their
    // data keeps the three protocols' steps aligned: a channel's share of a block that
    // fills a Simple slot fills an LL or LL128 slot too, rather than spilling a sliver into
    // a second slot that costs a whole handshake.
    const int proto = ringProto;
    p->proto = proto;
    size_t chunk = q->chunkBytes;
    if (chunk == 0) {
        // 1 MiB chunks, or smaller so that all FIFOs (2 chunks per (channel, rank), in wire
        // bytes) stay within 1 GiB.  Measured on GB300, large chunks win even when the FIFOs
        // do not fit in L2 (the slots in flight mostly stay there, being kept ahead of the
        // user data), while L2-sized chunks (64-128 KiB at 32 channels) spend the time in
        // the per-slot handshake (8 x 64 MiB, 32 channels, Simple: 428 us with 1 MiB chunks
        // against 627 us with 128 KiB).
        size_t fit = ((size_t)1 << 30) / (2 * (size_t)q->nChannels * (size_t)N);   // wire bytes per chunk
        if (proto == vProtoLL) fit /= 2;
        else if (proto == vProtoLL128) fit = fit / 128 * 120;
        chunk = std::min<size_t>((size_t)1 << 20, std::max<size_t>(16384, pow2_floor(fit)));
        // Broadcast passes a channel's whole share (D bytes) down a chain of N-1 hops in k
        // slots, which takes about (N - 2 + k) (h + D / (k R)) for a per-slot handshake h
        // and a per-CTA rate R; the best k is sqrt((N - 2) D / (h R)).  With h R about
        // 40 KB on GB300 (2 us at 20 GB/s), the slot is D / k rounded up to a power of two,
        // between 1 KiB and a quarter of the chunk.  (For the ring collectives every step
        // moves another block, and large slots, which amortise the handshake, win.)
        if (q->coll == vCollBroadcast && N > 2) {
            const double share = (double)(std::min(p->channelElems, B) * esz);
            const double k = std::max(1.0, std::sqrt((double)(N - 2) * share / 40960.0));
            size_t slot = 1024;
            while ((double)slot < share / k && slot * vc::kChunkSlots < chunk) slot *= 2;
            chunk = slot * vc::kChunkSlots;
        }
    }
    const size_t slotPayload = chunk / vc::kChunkSlots;   // >= 1 KiB, a power of two
    size_t slotBytes = slotPayload;
    if (proto == vProtoLL) slotBytes = 2 * slotPayload;
    else if (proto == vProtoLL128) slotBytes = align_up(div_up(slotPayload, (size_t)120), 2) * 128;
    p->slotBytes = slotBytes;
    p->slotPayloadElems = slotPayload / esz;
    p->chunkElems = p->slotPayloadElems * vc::kChunkSlots;
    p->fifoBytes = slotBytes * vc::kFifoSlots;
    p->nChannels = q->nChannels;
    p->ctasPerChannel = N;
    p->gridCtas = N * q->nChannels;
    // Threads per (channel, rank) CTA: the per-protocol thread thresholds (NCCL book
    // section 2.4, comm.h: LL 8, LL128 8, Simple 64), read as the fewest payload bytes of
    // one step that each thread should carry -- a small step runs on fewer threads (never
    // fewer than two warps), which makes the per-slot barriers cheaper.
    const size_t threshold = proto == vProtoSimple ? 64 : 8;
    const size_t stepBytes = std::min(p->chunkElems, std::max<size_t>(1, std::min(p->channelElems, B))) * esz;
    int nt = vc::kRingThreads;
    while (nt > 64 && stepBytes < (size_t)nt * threshold) nt /= 2;
    p->threadsPerCta = nt;
    // The 16-byte path of the ring also needs every slot and chunk to start on a vector.
    if (p->slotPayloadElems % VE != 0) p->vectorized = 0;
    p->vecBytes = p->vectorized ? 16 : 0;
    return vSuccess;
}

extern "C" vResult_t vPlanChannelRange(const vPlanInfo_t* p, size_t count, int channel, int block,
                                       size_t* lo, size_t* hi) {
    if (!p || !lo || !hi || channel < 0 || channel >= p->nChannels || block < 0) return vInvalidArgument;
    const size_t base = (size_t)block * p->blockElems;
    size_t l = base + std::min((size_t)channel * p->channelElems, p->blockElems);
    size_t h = base + std::min((size_t)(channel + 1) * p->channelElems, p->blockElems);
    l = std::min(l, count);
    h = std::min(h, count);
    *lo = l;
    *hi = std::max(l, h);
    return vSuccess;
}

extern "C" vResult_t vPlanTreeLinks(int nRanks, int rank, int tree, int* parent, int* child0, int* child1) {
    if (nRanks < 1 || nRanks > VCOMM_MAX_RANKS || rank < 0 || rank >= nRanks || (tree != 0 && tree != 1) ||
        !parent || !child0 || !child1)
        return vInvalidArgument;
    // Binary tree over ranks 0..n-1 (NCCL book chapter 4, ncclGetBtree): the lowest set bit
    // of a rank is its level's step; rank 0 (no bit in range) is the root.
    auto btree = [nRanks](int r, int* u, int* a, int* b) {
        int step = 1;
        while (step < nRanks && (r & step) == 0) step <<= 1;
        if (r == 0) {
            *u = -1;
            *a = -1;
            *b = nRanks > 1 ? step / 2 : -1;
            return;
        }
        int up = (r ^ step) | (step << 1);
        *u = up < nRanks ? up : (r ^ step);
        int half = step / 2;
        *a = half > 0 ? r - half : -1;
        *b = -1;
        for (; half > 0; half /= 2)
            if (r + half < nRanks) { *b = r + half; break; }
    };
    if (tree == 0) {
        btree(rank, parent, child0, child1);
        return vSuccess;
    }
    // Second tree (ncclGetDtree): the first one mirrored for an even count, shifted by one
    // rank for an odd count.
    int u, a, b;
    const bool mirror = nRanks % 2 == 0;
    btree(mirror ? nRanks - 1 - rank : (rank + nRanks - 1) % nRanks, &u, &a, &b);
    auto map = [&](int x) { return x < 0 ? -1 : (mirror ? nRanks - 1 - x : (x + 1) % nRanks); };
    *parent = map(u);
    *child0 = map(a);
    *child1 = map(b);
    return vSuccess;
}
