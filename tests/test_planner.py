"""Host planner (vPlanCompute / vPlanChannelRange), no GPU needed."""
from __future__ import annotations

import os

import pytest

import oracle
from collective_communication_virtual_gb300 import build, vcomm as V

ESZ = {V.vFloat32: 4, V.vFloat16: 2, V.vBFloat16: 2, V.vInt32: 4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    V.lib()


def plan(**kw):
    req = dict(nRanks=8, nChannels=1, proto=V.vProtoSimple, algo=V.vAlgoAuto, coll=V.vCollAllReduce,
               datatype=V.vFloat32, count=1024, chunkBytes=0, aligned16=1, smCount=152,
               l2Bytes=126 << 20, aligned32=0)
    req.update(kw)
    return V.vPlanCompute(**req)


def covered(p, total, nblocks, nch):
    seen = bytearray(total)
    for ch in range(nch):
        for b in range(nblocks):
            lo, hi = V.vPlanChannelRange(p, total, ch, b)
            for e in range(lo, hi):
                assert not seen[e], (ch, b, e)
                seen[e] = 1
    return all(seen)


@pytest.mark.parametrize("dt", [V.vFloat32, V.vBFloat16])
def test_allreduce_partition_covers_every_element_once(dt):
    for n in (1, 2, 3, 4, 7, 8):
        for count in (0, 1, 5, 17, 1000, 4099, 65_537):
            for nch in (1, 2, 3, 8, 16):
                p = plan(nRanks=n, nChannels=nch, count=count, datatype=dt)
                assert p.blockElems == oracle.block_elems(count, n, ESZ[dt])
                assert covered(p, count, n, nch), (n, count, nch)


def test_allreduce_blocks_and_channel_ranges_start_on_16_bytes():
    for dt in (V.vFloat32, V.vFloat16):
        for n, count, nch in [(8, 16 << 20, 32), (3, 100_003, 5), (8, 4099, 16)]:
            p = plan(nRanks=n, nChannels=nch, count=count, datatype=dt)
            for ch in range(nch):
                for b in range(n):
                    lo, hi = V.vPlanChannelRange(p, count, ch, b)
                    if hi > lo:
                        assert (lo * ESZ[dt]) % 16 == 0


def test_reduce_scatter_and_copies_partition():
    for coll, nblocks in [(V.vCollReduceScatter, None), (V.vCollAllGather, None),
                          (V.vCollBroadcast, 1)]:
        for n, count, nch in [(8, 4096, 8), (5, 3001, 3), (2, 1, 4)]:
            p = plan(coll=coll, nRanks=n, nChannels=nch, count=count, noBulkCopy=1)
            nb = nblocks or n
            assert covered(p, count * nb, nb, nch)


def test_vector_path_requires_aligned_blocks():
    assert plan(coll=V.vCollReduceScatter, count=4096).vectorized == 1
    assert plan(coll=V.vCollReduceScatter, count=4097).vectorized == 0
    assert plan(coll=V.vCollAllReduce, count=4097).vectorized == 1      # only the tail is ragged
    assert plan(coll=V.vCollAllReduce, count=4096, aligned16=0).vectorized == 0
    assert plan(coll=V.vCollAllGather, count=8, datatype=V.vBFloat16).vectorized == 1
    assert plan(coll=V.vCollAllGather, count=12, datatype=V.vBFloat16).vectorized == 0


def test_ring_geometry_follows_the_step_constants():
    # A chunk is 4 slots of chunk / 4 data bytes; a slot's wire size follows the protocol:
    # the data itself (Simple), a 4-byte flag per 4 data bytes (LL), 120 data bytes per
    # 128-byte line, an even number of lines (LL128).
    for proto, wire in [(V.vProtoSimple, 256 << 10), (V.vProtoLL, 512 << 10),
                        (V.vProtoLL128, (-(-(256 << 10) // 120) + 1) // 2 * 2 * 128)]:
        p = plan(algo=V.vAlgoRing, proto=proto, count=1 << 24, chunkBytes=1 << 20)
        assert p.algo == V.vAlgoRing and p.proto == proto
        assert p.slotPayloadElems * 4 * 4 == 1 << 20      # a chunk is 4 slots of data
        assert p.chunkElems == 4 * p.slotPayloadElems
        assert p.slotBytes == wire
        assert p.fifoBytes == 8 * p.slotBytes             # NCCL_STEPS = 8
        assert p.gridCtas == 8 and p.ctasPerChannel == 8
    ll128 = plan(algo=V.vAlgoRing, proto=V.vProtoLL128, count=1 << 24, chunkBytes=1 << 20)
    assert ll128.slotBytes // 128 * 120 >= ll128.slotPayloadElems * 4 > (ll128.slotBytes // 128 - 2) * 120


def test_default_chunk_is_1_mib_within_a_1_gib_fifo_budget():
    for n, nch in [(8, 1), (8, 8), (8, 32), (4, 64)]:
        for proto in (V.vProtoSimple, V.vProtoLL, V.vProtoLL128):
            p = plan(algo=V.vAlgoRing, proto=proto, nRanks=n, nChannels=nch, count=1 << 26)
            chunk = p.chunkElems * 4
            assert p.fifoBytes * n * nch <= 1 << 30
            if proto != V.vProtoLL or n * nch <= 256:
                assert chunk == 1 << 20
            else:
                assert chunk == 512 << 10
    p = plan(algo=V.vAlgoRing, nRanks=64, nChannels=64, count=1 << 26)
    assert p.chunkElems * 4 == 128 << 10 and p.fifoBytes * 64 * 64 <= 1 << 30


def test_auto_protocol_follows_the_fitted_ring_model():
    # 32 channels: LL has the lowest latency, Simple the highest bus bandwidth
    small = plan(algo=V.vAlgoRing, proto=V.vProtoAuto, count=256, nChannels=32)       # 1 KiB
    big = plan(algo=V.vAlgoRing, proto=V.vProtoAuto, count=16 << 20, nChannels=32)    # 64 MiB
    assert (small.proto, big.proto) == (V.vProtoLL, V.vProtoSimple)
    # the prediction is the smallest of the three protocols
    for count in (256, 1 << 18, 1 << 20, 16 << 20):
        auto = plan(algo=V.vAlgoRing, proto=V.vProtoAuto, count=count, nChannels=8)
        each = [plan(algo=V.vAlgoRing, proto=p, count=count, nChannels=8).predictedUs for p in range(3)]
        assert auto.predictedUs == pytest.approx(min(each))


def test_model_evaluates_its_fitted_constants():
    # fp32 all-reduce, 8 ranks: one-pass 1.5 us + minimum bytes / 7.097e6 B/us; the staged
    # ring with Simple at 32 channels: 36.88 us + 5.87 us per MiB up to the 64 MiB knee +
    # the rest / 136493.1 B/us; at 1 channel 32.78 us + 94.19 us per MiB up to 512 KiB +
    # the rest / 8645.7 B/us
    mib = 1 << 20
    big = 256 * mib
    assert plan(count=256).predictedUs == pytest.approx(1.5 + 16 * 1024 / 7.097e6, rel=0.001)
    assert plan(count=64 << 20).predictedUs == pytest.approx(1.5 + 16 * big / 7.097e6, rel=0.001)
    assert plan(algo=V.vAlgoRing, count=256, nChannels=32).predictedUs == \
        pytest.approx(36.88 + 5.87 * 1024 / mib, rel=1e-4)
    assert plan(algo=V.vAlgoRing, count=64 << 20, nChannels=32).predictedUs == \
        pytest.approx(36.88 + 5.87 * 64 + (big - 64 * mib) / 136493.1, rel=1e-4)
    assert plan(algo=V.vAlgoRing, count=64 << 20, nChannels=1).predictedUs == \
        pytest.approx(32.78 + 94.19 / 2 + (big - mib // 2) / 8645.7, rel=1e-4)


def test_auto_algorithm_picks_the_one_pass_kernels():
    for count in (256, 1 << 16, 1 << 22, 1 << 26):
        for nch in (1, 8, 32):
            p = plan(algo=V.vAlgoAuto, count=count, nChannels=nch, proto=V.vProtoAuto)
            assert p.algo == V.vAlgoOnePass
            assert p.predictedUs < plan(algo=V.vAlgoRing, count=count, nChannels=nch,
                                        proto=V.vProtoAuto).predictedUs


def test_prediction_grows_with_size_and_channels_help_the_ring():
    prev = 0
    for k in range(11):
        t = plan(algo=V.vAlgoRing, count=256 * 4 ** k, nChannels=8).predictedUs
        assert t > prev
        prev = t
    big = 16 << 20
    assert plan(algo=V.vAlgoRing, count=big, nChannels=32).predictedUs < \
        plan(algo=V.vAlgoRing, count=big, nChannels=1).predictedUs


def test_one_rank_and_alltoall_always_one_pass():
    assert plan(nRanks=1, algo=V.vAlgoRing).algo == V.vAlgoOnePass
    assert plan(coll=V.vCollAllToAll, algo=V.vAlgoRing).algo == V.vAlgoOnePass
    assert plan(coll=V.vCollAllToAllv, algo=V.vAlgoRing).algo == V.vAlgoOnePass


def test_traffic_and_bus_factor():
    n, count = 8, 16 << 20
    S = count * 4
    p = plan(nRanks=n, count=count)
    assert p.minBytes == 2 * n * S and p.busFactor == pytest.approx(2 * (n - 1) / n)
    p = plan(nRanks=n, count=count, coll=V.vCollReduceScatter)
    assert p.minBytes == n * n * S + n * S and p.busFactor == pytest.approx((n - 1) / n)
    p = plan(nRanks=n, count=count, coll=V.vCollAllGather)
    assert p.minBytes == n * S + n * n * S
    p = plan(nRanks=n, count=count, coll=V.vCollBroadcast)
    assert p.minBytes == S + n * S
    p = plan(nRanks=n, count=count, coll=V.vCollAllToAll)
    assert p.minBytes == 2 * n * n * S
    p = plan(nRanks=n, count=count, coll=V.vCollReduce)
    assert p.minBytes == n * S + S and p.blockElems == oracle.block_elems(count, n, 4)
    assert plan(nRanks=n, count=count, coll=V.vCollGather).minBytes == 2 * n * S
    assert plan(nRanks=n, count=count, coll=V.vCollScatter).minBytes == 2 * n * S
    assert plan(nRanks=n, count=count, coll=V.vCollReduce, algo=V.vAlgoRing).algo == V.vAlgoOnePass


def test_32_byte_vectors_when_blocks_and_pointers_allow():
    # B = 2M fp32 elements (8 MiB): a multiple of 32 bytes
    p = plan(count=16 << 20, aligned32=1)
    # flat grid: one 256-thread CTA per 256 vectors of every rank (2M / 8 / 256 = 1024 per
    # block, 8 blocks); the persistent grid is one 512-thread CTA per SM
    assert p.vecBytes == 32 and p.threadsPerCta == 256 and p.gridCtas == 8192
    assert plan(count=16 << 20, aligned32=1, persistentGrid=1).gridCtas == 152
    assert plan(count=16 << 20, aligned32=0).vecBytes == 16
    # B = alignUp(513, 4) = 516 elements = 2064 bytes: 16-byte blocks only
    assert plan(count=4099, aligned32=1).vecBytes == 16
    assert plan(count=4099, aligned16=0, aligned32=0).vecBytes == 0
    assert plan(coll=V.vCollReduceScatter, count=4096, aligned32=1).vecBytes == 32
    assert plan(coll=V.vCollAllGather, count=4096, aligned32=1).vecBytes == 32
    assert plan(coll=V.vCollAllGather, count=1 << 24, aligned32=1, noBulkCopy=1).gridCtas == 8 * 1024  # 64 KiB tiles
    assert plan(coll=V.vCollAllGather, count=1 << 24, aligned32=1, noBulkCopy=1, persistentGrid=1).gridCtas == 2 * 152


def test_tree_programs_fit_the_run_time_kernels_stack():
    # The run-time tree kernel keeps the newest partial in registers and the partials
    # waiting for their parent on a shared-memory stack of 8 entries per thread.  Walk
    # both trees' post-order programs for every rank count up to 64 and bound that stack.
    worst = 0
    for n in range(1, 65):
        for t in range(2):
            links = {v: V.vPlanTreeLinks(n, v, t) for v in range(n)}
            roots = [v for v in range(n) if links[v][0] < 0]
            assert len(roots) == 1
            prog = []

            def visit(v):
                kids = [k for k in links[v][1:] if k >= 0]
                for k in kids:
                    visit(k)
                prog.append(len(kids))

            visit(roots[0])
            assert len(prog) == n
            below = 0                 # partials below the register-held top
            for i, c in enumerate(prog):
                if c == 2:
                    below -= 1
                elif c == 0 and i > 0:
                    below += 1
                assert below >= 0
                worst = max(worst, below)
    assert worst <= 8, worst


def test_element_path_threads_take_8_elements_of_every_rank():
    # pointers off 16 bytes: no vectors; one thread per 8 elements of every rank
    p = plan(count=1 << 20, aligned16=0)                       # B = 131,072
    assert p.vecBytes == 0 and p.threadsPerCta == 256
    assert p.gridCtas == (131_072 // 8) * 8 // 256
    # a ragged reduce-scatter block of 1,048,577 fp32 elements, 8 ranks: 131,073 threads per
    # block; of bf16, warp tiles of 16-byte vectors, one per thread: 131,073 as well
    p = plan(coll=V.vCollReduceScatter, count=(1 << 20) + 1)
    assert p.vecBytes == 0 and p.threadsPerCta == 128
    assert p.gridCtas == -(-131_073 * 8 // 128)
    p = plan(coll=V.vCollReduceScatter, count=(1 << 20) + 1, datatype=V.vBFloat16)
    assert p.gridCtas == -(-131_073 * 8 // 128)
    # 3 ranks: four vectors per thread, 1,536 CTAs of work, under two waves of 1,216, so
    # one wave strides over it; 6 ranks keep the 8-element warp tiles
    p = plan(coll=V.vCollReduceScatter, nRanks=3, count=(1 << 20) + 1)
    assert p.gridCtas == 2 * 152 * (512 // 128)
    p = plan(coll=V.vCollReduceScatter, nRanks=6, count=(1 << 20) + 1)
    assert p.gridCtas == -(-131_073 * 6 // 128)


def test_copy_threads_follow_how_often_a_loaded_byte_is_stored():
    # 8 MiB blocks, 8 ranks.  All-gather and broadcast store every loaded byte 8 times: 32
    # bytes of a tile per thread (capped at 512 threads); their tiles halve to 8 KiB while
    # there are fewer than 16 per SM (all-gather: 16 KiB, 4096 tiles; broadcast, one block:
    # 8 KiB).  Gather, scatter and all-to-all store it once: 128 bytes per thread.
    p = plan(coll=V.vCollAllGather, count=1 << 21, aligned32=1, noBulkCopy=1)
    assert p.tileBytes == 16384 and p.threadsPerCta == 512
    p = plan(coll=V.vCollBroadcast, count=1 << 21, aligned32=1, noBulkCopy=1)
    assert p.tileBytes == 8192 and p.threadsPerCta == 256 and p.gridCtas == 1024
    # the FSDP bucket's all-gather: 3.125 MiB bf16 blocks -> 8 KiB tiles, 3200 CTAs
    p = plan(coll=V.vCollAllGather, count=1_638_400, datatype=V.vBFloat16, aligned32=1, noBulkCopy=1)
    assert p.tileBytes == 8192 and p.threadsPerCta == 256 and p.gridCtas == 3200
    for coll in (V.vCollGather, V.vCollScatter):
        p = plan(coll=coll, count=1 << 21, aligned32=1, noBulkCopy=1)
        assert p.tileBytes == 32768 and p.threadsPerCta == 256 and p.gridCtas == 2048
    # all-to-all, 4 MiB per rank: 64 blocks of 512 KiB -> 16 KiB tiles of 128 threads
    p = plan(coll=V.vCollAllToAll, count=(4 << 20) // 8 // 4, aligned32=1)
    assert p.tileBytes == 16384 and p.threadsPerCta == 128 and p.gridCtas == 2048
    # the persistent shape keeps 64 KiB tiles and 512-thread CTAs
    p = plan(coll=V.vCollAllToAll, count=(4 << 20) // 8 // 4, aligned32=1, persistentGrid=1)
    assert p.tileBytes == 65536 and p.threadsPerCta == 512


def test_fanout_copies_use_tma_bulk_copies_when_blocks_allow():
    p = plan(coll=V.vCollAllGather, count=1 << 21)                   # 8 MiB blocks
    # flat: one 16 KiB tile per single-stage CTA (512 tiles per block, 8 blocks)
    assert p.bulkCopy == 1 and p.threadsPerCta == 32 and p.tmaStages == 1 and p.gridCtas == 4096
    # persistent: three 4-stage CTAs per SM
    p = plan(coll=V.vCollAllGather, count=1 << 21, persistentGrid=1)
    assert p.bulkCopy == 1 and p.tmaStages == 4 and p.gridCtas == 3 * 152
    p = plan(coll=V.vCollBroadcast, count=4096)                      # 16 KiB: one tile
    assert p.bulkCopy == 1 and p.gridCtas == 1
    assert plan(coll=V.vCollGather, count=1 << 20).bulkCopy == 1
    assert plan(coll=V.vCollBroadcast, count=4097).bulkCopy == 0     # not a multiple of 16 bytes
    assert plan(coll=V.vCollAllGather, count=1 << 20, aligned16=0).bulkCopy == 0
    assert plan(coll=V.vCollAllGather, count=1 << 20, noBulkCopy=1).bulkCopy == 0
    assert plan(coll=V.vCollAllToAll, count=1 << 20).bulkCopy == 0
    assert plan(coll=V.vCollAllGather, count=4100, aligned32=1).vecBytes == 16
    for n, count, nch in [(8, 16 << 20, 32), (3, 100_003, 5)]:
        p = plan(nRanks=n, nChannels=nch, count=count)
        assert (p.channelElems * 4) % 32 == 0


def test_flat_grid_covers_the_work_once_and_persistent_grid_is_one_wave():
    # flat (default): one 256-thread CTA per 256 units (a 16-byte vector of every rank)
    p = plan(count=16 << 20, nChannels=1)
    assert p.vecBytes == 16 and p.threadsPerCta == 256 and p.gridCtas == (16 << 20) // 4 // 256
    p = plan(count=16 << 20, nChannels=32)
    assert p.nChannels * p.ctasPerChannel == p.gridCtas
    assert p.ctasPerChannel * 256 * 4 >= (16 << 20) // 32              # every unit has a thread
    assert (p.ctasPerChannel - 1) * 256 * 4 < (16 << 20) // 32         # and no CTA is idle
    # reduce-scatter: 128-thread CTAs
    p = plan(coll=V.vCollReduceScatter, count=2 << 20, aligned32=1)
    assert p.threadsPerCta == 128 and p.gridCtas == (16 << 20) // 8 // 128
    # persistent: about two resident 512-thread CTAs per SM, one wave, nearly full
    p = plan(count=16 << 20, nChannels=1, persistentGrid=1)
    assert p.gridCtas == 2 * 152
    p = plan(count=16 << 20, nChannels=32, persistentGrid=1)
    assert p.nChannels * p.ctasPerChannel == p.gridCtas
    assert 2 * 152 - 32 < p.gridCtas <= 2 * 152
    for persistent in (0, 1):
        assert plan(count=256, persistentGrid=persistent).gridCtas == 1   # 1 KiB per rank


def test_bad_requests():
    for kw in [dict(nRanks=0), dict(nRanks=65), dict(nChannels=0), dict(nChannels=65), dict(coll=9),
               dict(datatype=7), dict(proto=5), dict(algo=5), dict(chunkBytes=1000), dict(coll=10),
               dict(chunkBytes=3 << 20)]:
        with pytest.raises(V.VcommError) as e:
            plan(**kw)
        assert e.value.code == V.vInvalidArgument


def test_tree_links_match_the_pages_example_and_the_oracle(golden_dir):
    # NCCL book ncclGetBtree worked example: rank 1 of 8 is a leaf under rank 2
    with open(os.path.join(golden_dir, "btree_rank1_n8.txt")) as f:
        row = [l for l in f if l.strip() and not l.startswith("#")][0].split()
    n, rank, parent, c0, c1 = map(int, row)
    assert V.vPlanTreeLinks(n, rank, 0) == (parent, c0, c1)
    for n in range(1, 65):
        for t in (0, 1):
            for r in range(n):
                assert V.vPlanTreeLinks(n, r, t) == oracle.tree_links(n, r, t), (n, t, r)


def test_tree_links_match_the_hand_worked_table(golden_dir):
    with open(os.path.join(golden_dir, "btree_links.txt")) as f:
        rows = [list(map(int, l.split())) for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 60
    for n, tree, rank, parent, c0, c1 in rows:
        assert V.vPlanTreeLinks(n, rank, tree) == (parent, c0, c1), (n, tree, rank)


def test_tree_plan():
    p = plan(algo=V.vAlgoTree, count=16 << 20)
    assert p.algo == V.vAlgoTree and p.blockElems == 8 << 20
    # grid = one wave of resident CTAs: one per SM for the register-held 8-rank 32-byte
    # kernel, two per SM otherwise
    # flat (default): one 512-thread CTA per 512 vectors of every rank
    wide = plan(algo=V.vAlgoTree, count=16 << 20, aligned32=1)
    assert wide.vecBytes == 32 and wide.gridCtas == (16 << 20) // 8 // 512
    assert p.vecBytes == 16 and p.gridCtas == (16 << 20) // 4 // 512
    # persistent: one wave of resident CTAs
    wide = plan(algo=V.vAlgoTree, count=16 << 20, aligned32=1, persistentGrid=1)
    assert wide.vecBytes == 32 and wide.gridCtas == 152
    assert plan(algo=V.vAlgoTree, count=16 << 20, nRanks=4, aligned32=1, persistentGrid=1).gridCtas == 304
    assert plan(algo=V.vAlgoTree, count=16 << 20, persistentGrid=1).gridCtas == 304
    assert plan(algo=V.vAlgoTree, count=16 << 20, coll=V.vCollReduceScatter).algo == V.vAlgoOnePass
    assert plan(algo=V.vAlgoTree, count=100, nRanks=1).algo == V.vAlgoOnePass


def test_small_work_spreads_over_more_smaller_ctas():
    # 16 KiB fp32 per rank, 8 ranks, 32-byte vectors: 512 units -> 64-thread CTAs, 8 of them
    p = plan(count=4096, aligned32=1)
    assert p.threadsPerCta == 64 and p.gridCtas == 8
    # 256 KiB: 8192 units -> 64-thread CTAs (128 of them, still fewer than the 152 SMs at 128)
    p = plan(count=65536, aligned32=1)
    assert p.threadsPerCta == 64 and p.gridCtas == 128
    # enough work for every SM: the all-reduce's default 256-thread CTAs
    p = plan(count=16 << 20, aligned32=1)
    assert p.threadsPerCta == 256
    # copies: tiles shrink to 2 KiB and CTAs to tile / 32 threads until every SM has a tile
    p = plan(coll=V.vCollAllGather, count=1024, aligned32=1, noBulkCopy=1)     # 4 KiB blocks
    assert p.tileBytes == 2048 and p.threadsPerCta == 64 and p.gridCtas == 2 * 8
    p = plan(coll=V.vCollAllGather, count=1 << 20, aligned32=1, noBulkCopy=1)  # 4 MiB blocks
    assert p.tileBytes == 8192 and p.threadsPerCta == 256                     # 4096 tiles
    # the persistent shape keeps 512-thread CTAs and 64 KiB tiles
    p = plan(count=4096, aligned32=1, persistentGrid=1)
    assert p.threadsPerCta == 512


def test_ring_threads_follow_the_protocol_thread_thresholds():
    # comm.h thresholds: Simple 64, LL 8, LL128 8 bytes of a step per thread
    big = plan(algo=V.vAlgoRing, proto=V.vProtoSimple, count=16 << 20, chunkBytes=1 << 20)
    assert big.threadsPerCta == 512
    # 1 KiB per rank: 128-byte blocks -> the floor of two warps for every protocol
    for proto in (V.vProtoSimple, V.vProtoLL, V.vProtoLL128):
        assert plan(algo=V.vAlgoRing, proto=proto, count=256).threadsPerCta == 64
    # 16 KiB per rank, one channel: 2 KiB steps -> Simple wants 32 threads (floor 64), LL 256
    assert plan(algo=V.vAlgoRing, proto=V.vProtoSimple, count=4096).threadsPerCta == 64
    assert plan(algo=V.vAlgoRing, proto=V.vProtoLL, count=4096).threadsPerCta == 256


def test_every_plan_is_launchable():
    # Sweep collectives, rank counts, channel counts, sizes, types, alignment and grid
    # shape: every plan must describe a launch the kernels accept.
    colls = [V.vCollAllReduce, V.vCollReduceScatter, V.vCollAllGather, V.vCollBroadcast, V.vCollAllToAll,
             V.vCollAllToAllv, V.vCollReduce, V.vCollGather, V.vCollScatter]
    counts = [1, 7, 1000, 4097, 65_536, 1_000_003, 1 << 24, (1 << 31) + 5]
    n_checked = 0
    for coll in colls:
        for n in (1, 2, 3, 8, 16, 64):
            for nch in (1, 3, 32):
                for count in counts:
                    for dt in (V.vFloat32, V.vBFloat16):
                        for a16, a32, persistent in ((1, 1, 0), (1, 0, 0), (0, 0, 0), (1, 1, 1)):
                            for algo in (V.vAlgoAuto, V.vAlgoRing, V.vAlgoTree):
                                p = plan(coll=coll, nRanks=n, nChannels=nch, count=count, datatype=dt,
                                         aligned16=a16, aligned32=a32, persistentGrid=persistent, algo=algo,
                                         noBulkCopy=1)
                                n_checked += 1
                                assert 1 <= p.gridCtas <= (1 << 30), (coll, n, nch, count)
                                assert p.threadsPerCta in (32, 64, 128, 256, 512), p.threadsPerCta
                                assert p.vecBytes in (0, 16, 32)
                                if not a16:
                                    assert p.vecBytes == 0
                                if not a32:
                                    assert p.vecBytes != 32
                                if p.algo == V.vAlgoRing:
                                    assert p.gridCtas == p.nChannels * n
                                    assert p.slotBytes >= 1024 and p.slotBytes % 256 == 0
                                    assert p.fifoBytes == 8 * p.slotBytes
                                    assert p.slotPayloadElems >= 1 and p.chunkElems >= p.slotPayloadElems
                                elif p.algo == V.vAlgoOnePass and coll in (V.vCollAllGather, V.vCollBroadcast,
                                                                           V.vCollAllToAll, V.vCollGather,
                                                                           V.vCollScatter):
                                    assert 2048 <= p.tileBytes <= 65_536
                                    assert p.tileBytes & (p.tileBytes - 1) == 0
                                if p.vecBytes and coll in (V.vCollAllReduce, V.vCollReduce):
                                    # all-reduce blocks follow alignUp(ceil(count/N), 16/esz), so a
                                    # vector never straddles two blocks
                                    esz = 4 if dt == V.vFloat32 else 2
                                    assert (p.blockElems * esz) % 16 == 0
    assert n_checked > 10_000
