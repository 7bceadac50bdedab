"""The host planner on made-up devices (pure function, no GPU)."""
import itertools
import random

import pytest

import sparse_attention_row_gb300 as sar
from sparse_attention_row_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def props(num_sms=152, occ=1, smem=217 * 1024, optin=227 * 1024, clusters=None, pair=(0, 0), small=(0, 0),
          short=(0, 0), short_clusters=None, short16=(0, 0), short16_clusters=None):
    """A made-up device; clusters (short_clusters) maps a cluster size to its co-resident count for
    the wide shape (the short-row kernel's cluster form), none by default; pair, small and short are
    (shared memory, CTAs per SM) of those shapes (absent by default)."""
    p = sar.TopkDeviceProps()
    p.num_sms, p.ctas_per_sm, p.smem_per_cta, p.max_smem_optin = num_sms, occ, smem, optin
    for c, n in (clusters or {}).items():
        p.cluster_groups[c] = n
    p.pair_smem_per_cta, p.pair_ctas_per_sm = pair
    p.small_smem_per_cta, p.small_ctas_per_sm = small
    p.short_smem_per_cta, p.short_ctas_per_sm = short
    for c, n in (short_clusters or {}).items():
        p.short_cluster_groups[c] = n
    p.short16_smem_per_cta, p.short16_ctas_per_sm = short16
    for c, n in (short16_clusters or {}).items():
        p.short16_cluster_groups[c] = n
    return p


GB300_SMALL = (85000, 2)


GB300_PAIR = (113536, 2)


GB300_SHORT = (220 * 1024, 1)


def gb300_clusters():
    # co-resident clusters of c CTAs of the kernel (one CTA per SM), as queried on a GB300
    return {2: 76, 3: 46, 4: 36, 5: 28, 6: 23, 7: 15, 8: 15}


def plan(p, rows, stride, next_n=1, topk=2048, **opt):
    o = sar.TopkOptions()
    for k, v in opt.items():
        setattr(o, k, v)
    return sar.topk_make_plan(p, rows, stride, next_n, topk, o)


def test_the_five_workloads_on_a_gb300():
    gb = props()
    rc, pl = plan(gb, 8, 4096, topk=512)
    assert rc == 0 and pl.ctas_per_group == 1 and pl.grid == 8 and not pl.cooperative
    rc, pl = plan(gb, 64, 32768)
    assert rc == 0 and pl.ctas_per_group == 1 and pl.grid == 64
    rc, pl = plan(gb, 16, 131072)
    assert rc == 0 and pl.ctas_per_group == 9 and pl.grid == 144 and pl.cooperative
    # two CTAs per row would save 81920 elements each, less than the merge costs
    rc, pl = plan(gb, 64, 163840, next_n=2, topk=1024)
    assert rc == 0 and pl.ctas_per_group == 1 and pl.grid == 64 and not pl.cooperative
    rc, pl = plan(gb, 4096, 65536)
    assert rc == 0 and pl.ctas_per_group == 1 and pl.grid == 152 and not pl.cooperative


def test_topk1024_mtp1_never_oversubscribes():
    # the deadlock case of the persistent kernel: long rows, TopK=1024, next_n=1
    for occ, sms in itertools.product((1, 2, 3), (20, 48, 132, 152, 160)):
        for rows in (1, 2, 3, 7, 16, 33, 64, 100, 1000, 5000):
            rc, pl = plan(props(num_sms=sms, occ=occ), rows, 200000, topk=1024)
            assert rc == 0
            if pl.cooperative:
                assert pl.grid <= sms * occ


def test_invariants_on_random_shapes():
    rng = random.Random(5)
    for _ in range(3000):
        sms, occ = rng.randint(1, 200), rng.randint(1, 4)
        rows = rng.choice([0, 1, 2, rng.randint(1, 64), rng.randint(1, 100000)])
        nn = rng.choice([1, 2, 4])
        rows -= rows % nn
        stride = rng.choice([1, 17, 4096, 32768, 32769, 131072, rng.randint(1, 1 << 22)])
        topk = rng.choice([512, 1024, 2048, 1, rng.randint(1, 4096)])
        force = rng.choice([0, 0, 0, 1, 2, 5, 16])
        maxc = rng.choice([0, 0, rng.randint(1, 400)])
        rc, pl = plan(props(num_sms=sms, occ=occ), rows, stride, next_n=nn, topk=topk,
                      force_ctas_per_group=force, max_ctas=maxc)
        cap = sms * occ if not maxc else min(sms * occ, maxc)
        if rc == sar.TOPK_ERR_PLAN:
            assert force > 1 and cap < force
            continue
        assert rc == 0
        G = pl.ctas_per_group
        assert 1 <= G <= 16
        if force:
            assert G == force
        assert pl.grid == pl.num_groups * G
        if rows == 0:
            assert pl.grid == 0
            continue
        assert 1 <= pl.num_groups <= rows
        if G > 1:
            assert pl.cooperative == 1
            assert pl.grid <= cap, (sms, occ, rows, stride, G)
            assert pl.num_groups <= sms
        else:
            assert pl.cooperative == 0 and pl.grid <= cap


def test_split_gain_rule():
    gb = props()
    for rows, stride in ((16, 131072), (4, 200000), (32, 96000), (64, 163840), (8, 65536), (2, 98304)):
        rc, pl = plan(gb, rows, stride)
        assert rc == 0
        G = pl.ctas_per_group
        if G > 1:
            assert stride * (G - 1) // G >= 90000
        else:
            g = min(16, 152 // rows, max(1, stride // 8192))
            assert g < 2 or stride <= 32768 or stride * (g - 1) // g < 90000


def test_cluster_plans_for_the_five_workloads():
    gb = props(clusters=gb300_clusters())
    # 16 rows: clusters of 7 or 8 would not all be resident (15 of them), so 6
    rc, pl = plan(gb, 16, 131072)
    assert rc == 0 and pl.ctas_per_group == 6 and pl.cluster and not pl.cooperative and pl.grid == 96
    rc, pl = plan(gb, 12, 131072)
    assert rc == 0 and pl.ctas_per_group == 8 and pl.cluster and pl.grid == 96
    rc, pl = plan(gb, 64, 163840, next_n=2, topk=1024)
    assert rc == 0 and pl.ctas_per_group == 2 and pl.cluster and pl.grid == 128
    rc, pl = plan(gb, 64, 32768)
    assert rc == 0 and pl.ctas_per_group == 1 and not pl.cluster
    rc, pl = plan(gb, 4096, 65536)
    assert rc == 0 and pl.ctas_per_group == 1 and not pl.cluster and pl.grid == 152
    # the workspace merge when asked for, and its own (larger) gain rule
    rc, pl = plan(gb, 16, 131072, merge=1)
    assert rc == 0 and pl.ctas_per_group == 9 and pl.cooperative and not pl.cluster
    rc, pl = plan(gb, 64, 163840, next_n=2, topk=1024, merge=1)
    assert rc == 0 and pl.ctas_per_group == 1


def test_cluster_forcing_and_limits():
    gb = props(clusters=gb300_clusters())
    rc, pl = plan(gb, 5, 100000, force_ctas_per_group=3)
    assert rc == 0 and pl.cluster and pl.grid == 15
    rc, pl = plan(gb, 5, 100000, force_ctas_per_group=3, merge=1)
    assert rc == 0 and not pl.cluster and pl.cooperative
    assert plan(gb, 5, 100000, force_ctas_per_group=9, merge=2)[0] == sar.TOPK_ERR_PLAN
    assert plan(props(), 5, 100000, force_ctas_per_group=2, merge=2)[0] == sar.TOPK_ERR_PLAN
    assert plan(gb, 5, 100000, merge=3)[0] == sar.TOPK_ERR_INVALID_ARG
    # a device without clusters falls back to the workspace merge by itself
    rc, pl = plan(props(), 16, 131072)
    assert rc == 0 and pl.ctas_per_group == 9 and not pl.cluster


def test_cluster_invariants_on_random_shapes():
    rng = random.Random(11)
    for _ in range(3000):
        sms, occ = rng.randint(8, 200), rng.randint(1, 2)
        cl = {c: rng.choice([0, rng.randint(1, sms // c)]) for c in range(2, 9)}
        rows = rng.choice([1, 2, rng.randint(1, 64), rng.randint(1, 5000)])
        stride = rng.choice([4096, 32769, 131072, rng.randint(1, 1 << 22)])
        force = rng.choice([0, 0, 2, 3, 8, 12])
        merge = rng.choice([0, 0, 1, 2])
        rc, pl = plan(props(num_sms=sms, occ=occ, clusters=cl), rows, stride, force_ctas_per_group=force,
                      merge=merge)
        if rc != 0:
            assert rc == sar.TOPK_ERR_PLAN
            assert force > 1 and (merge == 2 or force > sms * occ)
            continue
        G = pl.ctas_per_group
        if pl.cluster:
            assert 2 <= G <= 8 and merge != 1 and not pl.cooperative
            assert 1 <= pl.num_groups <= min(rows, cl[G])
        elif G > 1:
            assert pl.cooperative and merge != 2 and pl.grid <= sms * occ
        assert pl.grid == pl.num_groups * G


def test_paired_shape():
    gb = props(clusters=gb300_clusters(), pair=GB300_PAIR)
    rc, pl = plan(gb, 4096, 65536)  # prefill: 27 rows per SM
    assert rc == 0 and pl.shape == 2 and pl.ctas_per_group == 1 and pl.grid == 304 and pl.threads == 416
    assert pl.smem_bytes == GB300_PAIR[0] and not pl.cooperative and not pl.cluster
    rc, pl = plan(gb, 64, 32768)  # decode: one row per CTA, the wide shape
    assert rc == 0 and pl.shape == 1 and pl.grid == 64 and pl.threads == 800
    rc, pl = plan(gb, 4 * 152 - 1, 65536)
    assert rc == 0 and pl.shape == 1
    rc, pl = plan(gb, 4 * 152, 65536)
    assert rc == 0 and pl.shape == 2 and pl.grid == 304
    rc, pl = plan(gb, 8, 4096, topk=512, shape=2)  # forced
    assert rc == 0 and pl.shape == 2 and pl.grid == 8
    rc, pl = plan(gb, 4096, 65536, shape=1)
    assert rc == 0 and pl.shape == 1 and pl.grid == 152
    rc, pl = plan(gb, 4096, 65536, max_ctas=100)
    assert rc == 0 and pl.shape == 2 and pl.grid == 100
    # the paired shape never splits a row, and needs a device that holds two of it
    assert plan(gb, 16, 131072, shape=2, force_ctas_per_group=4)[0] == sar.TOPK_ERR_INVALID_ARG
    rc, pl = plan(gb, 16, 131072, shape=2)
    assert rc == 0 and pl.shape == 2 and pl.ctas_per_group == 1
    assert plan(props(), 8, 4096, shape=2)[0] == sar.TOPK_ERR_PLAN
    assert plan(gb, 8, 4096, shape=6)[0] == sar.TOPK_ERR_INVALID_ARG
    assert plan(gb, 8, 4096, shape=5)[0] == sar.TOPK_ERR_PLAN  # no 16-warp short-row kernel on this made-up device
    assert plan(gb, 8, 4096, shape=4)[0] == sar.TOPK_ERR_PLAN  # no short-row kernel on this made-up device
    assert plan(gb, 8, 4096, shape=3)[0] == sar.TOPK_ERR_PLAN  # no small shape on this made-up device
    # TopK above 2048 runs on the wide shape only
    rc, pl = plan(gb, 4096, 65536, topk=3000)
    assert rc == 0 and pl.shape == 1
    assert plan(gb, 8, 4096, topk=2049, shape=2)[0] == sar.TOPK_ERR_UNSUPPORTED_TOPK
    rc, pl = plan(gb, 4096, 65536, topk=777)
    assert rc == 0 and pl.shape == 2


def test_low_shared_memory_devices():
    # a GB10-class part: ~99 KB per block holds neither the wide nor the paired shape
    gb10 = props(num_sms=48, smem=224 * 1024, optin=99 * 1024, pair=(113536, 0), small=(85000, 1))
    gb10.ctas_per_sm = 0
    rc, pl = plan(gb10, 64, 32768)
    assert rc == 0 and pl.shape == 3 and pl.ctas_per_group == 1 and pl.grid == 48 and pl.threads == 288
    rc, pl = plan(gb10, 16, 131072)  # long rows are not split on the small shape
    assert rc == 0 and pl.shape == 3 and pl.ctas_per_group == 1 and not pl.cooperative
    assert plan(gb10, 8, 4096, topk=3000)[0] == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert plan(gb10, 8, 4096, shape=1)[0] == sar.TOPK_ERR_PLAN
    # a partition that holds the paired shape but not the wide one
    mig = props(optin=120 * 1024, pair=GB300_PAIR, small=GB300_SMALL)
    rc, pl = plan(mig, 64, 32768)
    assert rc == 0 and pl.shape == 2
    # the small shape forced on a full GB300
    gb = props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL)
    rc, pl = plan(gb, 64, 32768, shape=3)
    assert rc == 0 and pl.shape == 3 and pl.grid == 64
    assert plan(gb, 64, 163840, shape=3, force_ctas_per_group=2)[0] == sar.TOPK_ERR_INVALID_ARG


def test_rejections():
    gb = props()
    assert plan(gb, 8, 4096, topk=0)[0] == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert plan(gb, 8, 4096, topk=4097)[0] == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert plan(gb, 9, 4096, next_n=2)[0] == sar.TOPK_ERR_INVALID_ARG
    assert plan(gb, 8, 0)[0] == sar.TOPK_ERR_INVALID_ARG
    assert plan(gb, 8, 4096, force_ctas_per_group=17)[0] == sar.TOPK_ERR_INVALID_ARG
    # a device whose opt-in shared memory holds none of the shapes
    assert plan(props(optin=64 * 1024, pair=GB300_PAIR, small=GB300_SMALL), 8, 200000)[0] == sar.TOPK_ERR_PLAN
    assert plan(props(occ=0), 8, 4096)[0] == sar.TOPK_ERR_PLAN


def test_threshold_and_capacity_knobs():
    gb = props()
    rc, pl = plan(gb, 16, 131072, long_row_threshold=200000)
    assert rc == 0 and pl.ctas_per_group == 1
    rc, pl = plan(gb, 16, 400000, max_ctas=40)
    assert rc == 0 and pl.ctas_per_group == 2 and pl.grid <= 40
    rc, pl = plan(gb, 16, 131072, max_ctas=40)  # a 2-way split saves too little
    assert rc == 0 and pl.ctas_per_group == 1
    rc, pl = plan(gb, 3, 4096, force_ctas_per_group=4)
    assert rc == 0 and pl.grid == 12 and pl.cooperative


def test_static_scratch_capacity_is_reachable_on_larger_devices():
    """topk_ragged_static's fixed array holds 76 row-group areas: every split plan on a GPU of up
    to 152 SMs fits (G >= 2 leaves at most num_sms / 2 groups), and a larger device can need more,
    which that entry point refuses with TOPK_ERR_WORKSPACE_TOO_SMALL."""
    static_groups = 76
    for rows in range(1, 152):
        for stride in (65536, 262144, 1 << 20):
            rc, pl = plan(props(), rows, stride)
            assert rc == 0
            if pl.ctas_per_group > 1:
                assert pl.num_groups <= static_groups
    # 200 SMs, no clusters: 90 rows of 1M elements split two ways through the workspace
    rc, pl = plan(props(num_sms=200), 90, 1 << 20)
    assert rc == 0 and pl.ctas_per_group == 2 and not pl.cluster and pl.num_groups == 90 > static_groups


def test_short_row_kernel():
    """Whole rows take the short-row kernel where the device holds it (rows of up to 16 pieces
    stay resident in its ring, longer ones stream through it), except batches of at least four
    rows per SM of up to 16384 elements, which the paired shape streams, and TopK of half the
    row or more, which the wide shape selects; only very long rows are split across CTAs (the
    thresholds are the crossovers that bench.py --sweep measured on a GB300)."""
    gb = props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL, short=GB300_SHORT)
    for rows, stride, k in ((8, 4096, 512), (64, 32768, 2048), (1, 1, 1), (300, 6000, 2048), (16, 131072, 2048),
                            (64, 163840, 1024), (4096, 65536, 3000), (4096, 65536, 2048), (4096, 32768, 2048),
                            (608, 16385, 2048), (152, 8192, 1024), (64, 4097, 2048), (10, 1000, 2048),
                            (64, 2048, 1024), (152, 2048, 2047)):
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 1 and pl.threads == 1024, (rows, stride, k)
        assert pl.grid == min(rows, 152) and not pl.cooperative and not pl.cluster
    for rows, stride, k in ((4096, 16384, 2048), (608, 8192, 2048), (608, 4096, 512), (4096, 2048, 1024)):
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.shape == 2 and pl.ctas_per_group == 1, (rows, stride, k)
    for rows, stride, k in ((64, 4096, 2048), (300, 6000, 4096), (1, 4096, 4095)):
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.shape == 1 and pl.ctas_per_group == 1, (rows, stride, k)
    # rows of a million elements and more, few of them, are still split across CTAs
    rc, pl = plan(gb, 16, 1 << 21)
    assert rc == 0 and pl.shape == 1 and pl.ctas_per_group > 1
    # forcing: shape 4 takes any length, but one CTA per row
    rc, pl = plan(gb, 10, 32768, shape=4, max_ctas=3)
    assert rc == 0 and pl.shape == 4 and pl.grid == 3
    rc, pl = plan(gb, 10, 400000, shape=4)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 1
    # a forced split of the short-row kernel: one row per cluster, merged in the cluster
    assert plan(gb, 10, 30000, shape=4, force_ctas_per_group=2)[0] == sar.TOPK_ERR_PLAN  # no clusters here
    gbc = props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL, short=GB300_SHORT,
                short_clusters=gb300_clusters())
    for rows, g in ((10, 2), (16, 6), (300, 8), (1, 3)):
        rc, pl = plan(gbc, rows, 30000, shape=4, force_ctas_per_group=g)
        assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == g and pl.cluster and not pl.cooperative
        assert pl.num_groups == rows and pl.grid == rows * g and pl.threads == 1024
    assert plan(gbc, 10, 30000, shape=4, force_ctas_per_group=9)[0] == sar.TOPK_ERR_INVALID_ARG
    assert plan(gbc, 10, 30000, shape=4, force_ctas_per_group=2, merge=1)[0] == sar.TOPK_ERR_PLAN
    rc, pl = plan(gb, 10, 30000, force_ctas_per_group=2)
    assert rc == 0 and pl.shape == 1 and pl.ctas_per_group == 2
    # the wide shape forced: the split rule of that kernel applies
    rc, pl = plan(gb, 16, 131072, shape=1)
    assert rc == 0 and pl.shape == 1 and pl.cluster and pl.ctas_per_group == 6
    # a device that cannot hold it (GB10-class shared memory) never plans it
    gb10 = props(num_sms=48, smem=224 * 1024, optin=99 * 1024, pair=(113536, 0), small=(85000, 1),
                 short=(220 * 1024, 0))
    rc, pl = plan(gb10, 8, 4096, topk=512)
    assert rc == 0 and pl.shape == 3
    assert plan(gb10, 8, 4096, topk=512, shape=4)[0] == sar.TOPK_ERR_PLAN


def test_short_row_cluster_split():
    """Few rows of 65536 up to 2^20 elements are split over a thread-block cluster of the
    short-row kernel: the largest size up to 8 with rows x size within the SMs whose clusters
    are all resident at once (the crossover that bench.py --sweep measured on a GB300)."""
    gb = props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL, short=GB300_SHORT,
               short_clusters=gb300_clusters())
    for rows, stride, k, g in ((16, 131072, 2048, 6),   # long_coop: 8 and 7 hold only 15 clusters
                               (64, 163840, 1024, 2),   # mtp
                               (4, 65536, 2048, 8), (16, 65536, 2048, 6), (1, 500000, 512, 8),
                               (76, 131072, 2048, 2), (28, 100000, 2048, 5), (30, 100000, 2048, 4), (40, 100000, 2048, 3),
                               (64, 32768, 2048, 2), (16, 32768, 2048, 6)):  # decode_batch: a tie, measured
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == g and pl.cluster, (rows, stride, k, pl.ctas_per_group)
        assert pl.grid == rows * g and pl.num_groups == rows and not pl.cooperative and pl.threads == 1024
    # whole rows: shorter rows, enough rows for every SM, very long rows
    for rows, stride, k in ((64, 32767, 2048), (8, 4096, 512), (16, 16384, 2048), (77, 131072, 2048),
                            (4096, 65536, 2048)):
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.ctas_per_group == 1 and not pl.cluster, (rows, stride, k)
    # very long rows: split over clusters while each CTA's expected candidates (about 8400 on
    # rows of 2^21 at TopK 2048) stay within 4096, else the wide shape, split or whole
    rc, pl = plan(gb, 16, 1 << 21)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 6 and pl.cluster
    rc, pl = plan(gb, 64, 1 << 21)
    assert rc == 0 and pl.shape == 1 and pl.ctas_per_group == 2
    rc, pl = plan(gb, 64, 1 << 20)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 2 and pl.cluster
    rc, pl = plan(gb, 128, 1 << 20)
    assert rc == 0 and pl.shape == 1 and pl.ctas_per_group == 1
    rc, pl = plan(gb, 128, 1 << 18)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 1
    # whole rows beyond 2^18 elements, or whose expected candidates exceed 4096 (TopK 4096 of
    # 65536), take the wide shape; split over clusters they stay on the short-row kernel
    for rows, stride, k, shape, g in ((128, 1 << 20, 512, 1, 1), (128, 1 << 19, 512, 1, 1), (128, 65536, 4096, 1, 1),
                                      (64, 65536, 4096, 4, 2), (64, 1 << 19, 4096, 4, 2), (16, 1 << 21, 512, 4, 6),
                                      # rows resident in the ring stay whole whatever their candidates
                                      (152, 32768, 4096, 4, 1), (608, 16384, 4096, 4, 1)):
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.shape == shape and pl.ctas_per_group == g, (rows, stride, k, pl.shape, pl.ctas_per_group)
    # the short-row kernel forced: the same rule; one CTA per row forced, or the workspace merge
    # asked for: whole rows
    rc, pl = plan(gb, 16, 131072, shape=4)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 6
    for opt in (dict(force_ctas_per_group=1), dict(merge=1), dict(shape=4, force_ctas_per_group=1)):
        rc, pl = plan(gb, 16, 131072, **opt)
        assert rc == 0 and pl.ctas_per_group == 1 and not pl.cluster, opt
    # a cap on the CTAs bounds rows x size
    rc, pl = plan(gb, 16, 131072, max_ctas=64)
    assert rc == 0 and pl.ctas_per_group == 4 and pl.grid == 64
    # no clusters on the device: whole rows
    rc, pl = plan(props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL, short=GB300_SHORT),
                  16, 131072)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 1


def test_short_row_kernel_with_16_warps():
    """The 16-warp instance of the short-row kernel (shape 5) takes whole rows of up to 4096
    elements (16384 at TopK 512 or less) and every split over a cluster, where the device holds
    it; the 32-warp instance keeps the longer whole rows (the crossovers bench.py --sweep measured
    on a GB300)."""
    gb = props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL, short=GB300_SHORT,
               short_clusters=gb300_clusters(), short16=GB300_SHORT, short16_clusters=gb300_clusters())
    for rows, stride, k, shape, g in ((8, 4096, 512, 5, 1), (152, 2048, 1024, 5, 1), (64, 32768, 2048, 5, 2),
                                      (152, 32768, 2048, 4, 1),
                                      (64, 16384, 512, 5, 1), (64, 16384, 1024, 4, 1), (64, 16385, 512, 4, 1),
                                      (4096, 65536, 2048, 4, 1), (16, 131072, 2048, 5, 6), (64, 163840, 1024, 5, 2),
                                      (608, 4096, 512, 2, 1), (64, 4096, 2048, 1, 1)):
        rc, pl = plan(gb, rows, stride, topk=k)
        assert rc == 0 and pl.shape == shape and pl.ctas_per_group == g, (rows, stride, k, pl.shape, pl.ctas_per_group)
        if shape == 5:
            assert pl.threads == 512 and pl.cluster == (g > 1)
    # forced: the 16-warp instance whole or split, like shape 4
    rc, pl = plan(gb, 10, 30000, shape=5, force_ctas_per_group=3)
    assert rc == 0 and pl.shape == 5 and pl.ctas_per_group == 3 and pl.cluster and pl.grid == 30
    rc, pl = plan(gb, 152, 32768, shape=5)
    assert rc == 0 and pl.shape == 5 and pl.ctas_per_group == 1 and pl.grid == 152
    assert plan(gb, 10, 30000, shape=5, force_ctas_per_group=9)[0] == sar.TOPK_ERR_INVALID_ARG
    # rows whose share per CTA exceeds 98304 elements split on the 32-warp instance
    for rows, stride, shape, g in ((1, 1 << 20, 4, 8), (16, 1 << 21, 4, 6), (1, 524288, 5, 8), (64, 196608, 5, 2),
                                   (64, 196609, 4, 2)):
        rc, pl = plan(gb, rows, stride)
        assert rc == 0 and pl.shape == shape and pl.ctas_per_group == g, (rows, stride, pl.shape, pl.ctas_per_group)
    # a device without the 16-warp instance splits on the 32-warp one
    gb32 = props(clusters=gb300_clusters(), pair=GB300_PAIR, small=GB300_SMALL, short=GB300_SHORT,
                 short_clusters=gb300_clusters())
    rc, pl = plan(gb32, 16, 131072)
    assert rc == 0 and pl.shape == 4 and pl.ctas_per_group == 6
