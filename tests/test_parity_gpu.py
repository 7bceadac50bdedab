"""Bit-exact parity of libtopk's CUDA path with the CPU oracle (GPU only)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import Runner, assert_matches_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rn():
    return Runner()


SMALL = [("decode_small", 8), ("decode_batch", 16), ("long_coop", 4), ("mtp", 8), ("prefill", 24)]


@pytest.mark.parametrize("name,rows", SMALL)
def test_workloads_small_auto(rn, name, rows):
    w = workloads.make(name, rows)
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n)
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n, label=name)
    assert rn.workspace_clean()


@pytest.mark.parametrize("shape", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("name,rows", SMALL)
def test_workloads_small_other_shapes(rn, name, rows, shape):
    """Every CTA shape forced on every workload: the wide one (24 consumer warps), the paired one
    (two CTAs of 12 consumer warps per SM), the small, low-shared-memory one (8 consumer warps), and
    the short-row kernel with 32 or 16 warps (rows of up to 16 pieces resident, longer rows
    streamed through its ring of 16 slots; long rows of few-row batches split over clusters)."""
    w = workloads.make(name, rows)
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n, options=rn.options(shape=shape))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n, label=f"{name} shape={shape}")
    assert rn.workspace_clean()


@pytest.mark.parametrize("topk", [1, 7, 100, 1000, 2047, 2049, 3000, 4096])
@pytest.mark.parametrize("G,merge,shape", [(0, 0, 0), (0, 0, 2), (0, 0, 3), (3, 1, 0), (4, 2, 0), (0, 0, 4),
                                           (3, 0, 4), (0, 0, 5), (3, 0, 5)])
def test_runtime_topk(rn, topk, G, merge, shape):
    """TopK outside the pages' 512 / 1024 / 2048, on every path (paired and small shapes up to 2048)."""
    if shape in (2, 3) and topk > 2048:
        pytest.skip("the paired and small shapes serve TopK up to 2048")
    rng = np.random.default_rng(topk)
    S = 40000
    x = np.round(rng.standard_normal((12, S)) * 32).astype(np.float32) / 32  # heavy ties
    lens = rng.integers(0, S, 12, endpoint=True).astype(np.int32)
    lens[:4] = [0, topk - 1 if topk > 1 else 0, topk, S]
    got = rn.run(x, lens, topk, options=rn.options(force_ctas_per_group=G, merge=merge, shape=shape))
    assert_matches_oracle(x, lens, got, topk, label=f"K={topk} G={G} merge={merge} shape={shape}")
    assert rn.workspace_clean()


@pytest.mark.parametrize("layout", ["transposed", "every_third_column", "padded_rows"])
@pytest.mark.parametrize("G,merge,shape", [(0, 0, 0), (1, 0, 1), (1, 0, 2), (1, 0, 3), (3, 1, 0), (4, 2, 0),
                                           (1, 0, 4), (1, 0, 5)])
def test_strided_logits(rn, layout, G, merge, shape):
    """Views with a row pitch and a column stride: transposed, column-strided, padded rows."""
    torch = rn.torch
    sar = rn.sar
    rng = np.random.default_rng(hash(layout) % 1000 + G)
    R, L, K = 10, 20000, 1024
    x = (np.round(rng.standard_normal((R, L)) * 16) / 16).astype(np.float32)
    lens = rng.integers(0, L, R, endpoint=True).astype(np.int32)
    lens[:4] = [0, K - 1, K, L]
    if layout == "transposed":
        view = torch.from_numpy(np.ascontiguousarray(x.T)).to(rn.dev).t()
    elif layout == "every_third_column":
        big = np.full((R, 3 * L), np.nan, np.float32)
        big[:, ::3] = x
        view = torch.from_numpy(big).to(rn.dev)[:, ::3]
    else:
        big = np.full((R, L + 100), np.nan, np.float32)
        big[:, :L] = x
        view = torch.from_numpy(big).to(rn.dev)[:, :L]
    ln = torch.from_numpy(lens).to(rn.dev)
    out = torch.full((R, K), -7, dtype=torch.int32, device=rn.dev)
    opts = rn.options(force_ctas_per_group=G, merge=merge, shape=shape)
    rc = sar.topk_ragged_strided(view, view.stride(0), view.stride(1), L, ln, R, 1, K, out,
                                 rn.sel.workspace, None, opts)
    assert rc == sar.TOPK_OK, sar.topk_status_string(rc)
    torch.cuda.synchronize()
    assert rn.sel.status() == 0
    assert_matches_oracle(x, lens, out.cpu().numpy(), K, label=f"{layout} G={G} merge={merge} shape={shape}")
    assert rn.workspace_clean()


def test_selector_takes_views_and_two_dimensional_lengths(rn):
    """The binding's Selector: a strided view, and next_n from [requests, next_n] lengths."""
    torch = rn.torch
    w = workloads.make("mtp", 8)
    ln2 = torch.from_numpy(w.lengths.reshape(-1, 2)).to(rn.dev)
    x = torch.from_numpy(w.logits).to(rn.dev)
    got = rn.sel(x, ln2, w.topk).cpu().numpy()
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, 2, label="selector mtp")
    xt = torch.from_numpy(np.ascontiguousarray(w.logits.T)).to(rn.dev).t()
    got = rn.sel(xt, ln2, w.topk).cpu().numpy()
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, 2, label="selector transposed")


@pytest.mark.parametrize("name,rows,topk", [("decode_small", 8, 512), ("decode_batch", 6, 2048),
                                            ("mtp", 4, 1024), ("prefill", 6, 2048), ("decode_batch", 6, 3000),
                                            ("decode_small", 8, 1)])
def test_values_and_sorted_rows(rn, name, rows, topk):
    """topk_gather_sort: the selected values, and rows ordered exactly as the oracle orders them."""
    torch = rn.torch
    sar = rn.sar
    w = workloads.make(name, rows)
    x = torch.from_numpy(w.logits).to(rn.dev)
    ln = torch.from_numpy(w.lengths).to(rn.dev)
    R, S = w.logits.shape
    out = torch.full((R, topk), -7, dtype=torch.int32, device=rn.dev)
    assert sar.topk_ragged(x, S, ln, R, w.next_n, topk, out, rn.sel.workspace) == sar.TOPK_OK
    unsorted = out.clone()
    val = torch.zeros((R, topk), dtype=torch.float32, device=rn.dev)
    # values only: indices untouched
    assert sar.topk_gather_sort(x, S, 1, S, R, topk, out, val, sort=False) == sar.TOPK_OK
    torch.cuda.synchronize()
    assert torch.equal(out, unsorted)
    idx, v = out.cpu().numpy(), val.cpu().numpy()
    ok = idx >= 0
    assert np.array_equal(v[ok], w.logits[np.nonzero(ok)[0], idx[ok]]) and np.all(np.isneginf(v[~ok]))
    # sorted: element by element equal to the oracle's rows (value desc, index asc, -1 last)
    assert sar.topk_gather_sort(x, S, 1, S, R, topk, out, val, sort=True) == sar.TOPK_OK
    want, _ = oracle.topk_ragged(w.logits, w.lengths, topk, next_n=w.next_n)
    got = out.cpu().numpy()
    assert np.array_equal(got, want), f"{name}: first bad row {np.nonzero((got != want).any(1))[0][:3]}"
    v = val.cpu().numpy()
    ok = got >= 0
    assert np.array_equal(v[ok], w.logits[np.nonzero(ok)[0], got[ok]]) and np.all(np.isneginf(v[~ok]))


def test_sorted_rows_of_a_transposed_view_through_the_selector(rn):
    torch = rn.torch
    w = workloads.make("decode_batch", 6)
    xt = torch.from_numpy(np.ascontiguousarray(w.logits.T)).to(rn.dev).t()
    ln = torch.from_numpy(w.lengths).to(rn.dev)
    idx, val = rn.sel(xt, ln, w.topk, sort=True, values=True)
    want, _ = oracle.topk_ragged(w.logits, w.lengths, w.topk)
    got = idx.cpu().numpy()
    assert np.array_equal(got, want)
    ok = got >= 0
    assert np.array_equal(val.cpu().numpy()[ok], w.logits[np.nonzero(ok)[0], got[ok]])


# merge 1: the CTAs of a row merge through the workspace (grid barrier);
# merge 2: they form a thread-block cluster and merge in its shared memory
SPLITS = [(1, 0), (2, 1), (2, 2), (3, 1), (3, 2), (5, 2), (8, 2), (9, 1), (16, 1)]


@pytest.mark.parametrize("G,merge", SPLITS)
@pytest.mark.parametrize("name,rows", [("decode_batch", 6), ("long_coop", 3), ("mtp", 4), ("prefill", 4)])
def test_workloads_forced_split(rn, name, rows, G, merge):
    w = workloads.make(name, rows)
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n,
                 options=rn.options(force_ctas_per_group=G, merge=merge))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n, label=f"{name} G={G} merge={merge}")
    assert rn.workspace_clean()


@pytest.mark.parametrize("shape", [4, 5])
@pytest.mark.parametrize("G", [2, 3, 4, 6, 8])
@pytest.mark.parametrize("name,rows", [("decode_small", 8), ("decode_batch", 6), ("long_coop", 3), ("mtp", 4),
                                       ("prefill", 4)])
def test_workloads_short_row_cluster_split(rn, name, rows, G, shape):
    """Each row split over a thread-block cluster of G short-row CTAs (32 or 16 warps; CTA c
    takes window pieces c, c + G, ...), merged in the cluster's shared memory."""
    w = workloads.make(name, rows)
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n, options=rn.options(shape=shape, force_ctas_per_group=G))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n,
                          label=f"{name} short-row cluster G={G} shape={shape}")
    assert rn.workspace_clean()


@pytest.mark.parametrize("name", workloads.NAMES)
def test_workloads_full_size(rn, name):
    """Every row of the full workload, in the launch configuration the benchmark times."""
    w = workloads.make(name)
    got = rn.run(w.logits, w.lengths, w.topk, w.next_n)
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, w.next_n, label=name + " full")
    assert rn.workspace_clean()


def _edge_rows(S: int, K: int, rng) -> tuple[np.ndarray, np.ndarray]:
    rows, lens = [], []
    base = rng.standard_normal(S).astype(np.float32)
    for L in (0, 1, K - 1, K, K + 1, 2 * K + 3, S - 1, S):
        rows.append(base.copy())
        lens.append(L)
    rows.append(np.full(S, 0.75, np.float32)); lens.append(S)                   # all equal
    rows.append(np.where(rng.random(S) < 0.5, -0.0, 0.0).astype(np.float32)); lens.append(S)  # +-0 mix
    r = rng.standard_normal(S).astype(np.float32)
    r[rng.integers(0, S, 50)] = np.inf
    r[rng.integers(0, S, 50)] = -np.inf
    rows.append(r); lens.append(S - 3)                                           # +-inf inside
    d = (rng.integers(-40, 40, S).astype(np.float32) * np.float32(1e-45))
    rows.append(d); lens.append(S)                                               # subnormals
    rows.append(np.arange(S, dtype=np.float32)); lens.append(S - 5)              # increasing
    rows.append(-np.arange(S, dtype=np.float32)); lens.append(S)                 # decreasing
    neg = -np.abs(rng.standard_normal(S)).astype(np.float32)
    rows.append(neg); lens.append(S)                                             # all negative
    few = np.full(S, -1.0, np.float32)
    few[rng.choice(S, K // 2, replace=False)] = 2.0
    rows.append(few); lens.append(S)                                             # K/2 distinct winners, ties below
    return np.stack(rows), np.array(lens, np.int32)


@pytest.mark.parametrize("topk", [512, 1024, 2048])
@pytest.mark.parametrize("S", [4096, 9001, 40000])
@pytest.mark.parametrize("G,merge,shape", [(0, 0, 0), (1, 0, 1), (0, 0, 2), (0, 0, 3), (4, 1, 0), (4, 2, 0), (8, 2, 0),
                                           (0, 0, 4), (2, 0, 4), (5, 0, 4), (8, 0, 4), (0, 0, 5), (4, 0, 5)])
def test_edge_cases(rn, topk, S, G, merge, shape):
    # with G = 8 and K = 2048 the all-equal row keeps 8 x K candidates at one
    # key, more than the leader's buffer: the cluster merge hands over to the
    # workspace merge
    rng = np.random.default_rng(S + topk)
    x, lens = _edge_rows(S, topk, rng)
    got = rn.run(x, lens, topk, options=rn.options(force_ctas_per_group=G, merge=merge, shape=shape))
    assert_matches_oracle(x, lens, got, topk, label=f"edges S={S} K={topk} G={G} merge={merge} shape={shape}")
    assert rn.workspace_clean()


def _dense_cluster_rows(S: int, rng) -> np.ndarray:
    """Rows of N(0,1) with about 3000 of their elements in a narrow cluster around 4 (sd
    0.05, 0.15 or 0.3), the last three also rounded to multiples of 2^-12 (equal keys)."""
    rows = []
    for i in range(6):
        x = rng.standard_normal(S).astype(np.float32)
        m = rng.random(S) < 3000.0 / S
        x[m] = (4.0 + (0.05, 0.15, 0.3)[i % 3] * rng.standard_normal(int(m.sum()))).astype(np.float32)
        if i >= 3:
            x = (np.round(x * 4096.0) / 4096.0).astype(np.float32)
        rows.append(x)
    return np.stack(rows)


def _kth_bin_size(row: np.ndarray, K: int) -> int:
    """Elements of the row that share the K-th largest value's top 15 key bits (sign,
    exponent and 6 mantissa bits): the size of the K-th key's bin in a radix select."""
    u = row.view(np.uint32).astype(np.uint64)
    keys = np.where(u >> 31 == 1, (~u) & 0xFFFFFFFF, u | 0x80000000)
    kth = np.sort(keys)[::-1][K - 1]
    return int(np.count_nonzero(keys >> 17 == kth >> 17))


@pytest.mark.parametrize("S", [30000, 100000])
@pytest.mark.parametrize("shape,G", [(0, 0), (4, 0), (4, 2), (4, 6), (5, 0), (5, 3)])
def test_large_kth_key_bin(rn, S, shape, G):
    """Hundreds of elements share the K-th key's bin (a dense cluster): the selection
    splits that bin further before ranking; with equal keys inside it, by index."""
    rng = np.random.default_rng(S + shape)
    K = 2048
    x = _dense_cluster_rows(S, rng)
    lens = np.full(x.shape[0], S, np.int32)
    sizes = [_kth_bin_size(r, K) for r in x]
    assert any(192 < n <= 512 for n in sizes), sizes  # the data reach the split
    got = rn.run(x, lens, K, options=rn.options(shape=shape, force_ctas_per_group=G))
    assert_matches_oracle(x, lens, got, K, label=f"dense cluster S={S} shape={shape} G={G} bins {sizes}")
    assert rn.workspace_clean()


@pytest.mark.parametrize("S,K", [(4096, 1536), (4096, 2048), (6000, 2800), (8192, 4096), (40000, 4096)])
@pytest.mark.parametrize("shape,G", [(0, 0), (4, 0), (4, 3), (5, 0), (5, 2)])
def test_kth_key_far_from_the_threshold(rn, S, K, shape, G):
    """The K-th key lies many binades above the seed's threshold: a selected fraction
    near one half of N(0,1) rows (the K-th value near zero), and rows whose values near
    the K-th span tiny magnitudes of both signs."""
    rng = np.random.default_rng(S * 7 + K)
    rows = [rng.standard_normal(S).astype(np.float32) for _ in range(4)]
    r = -np.abs(rng.standard_normal(S)).astype(np.float32)
    pos = rng.random(S) < (K * 0.6) / S
    r[pos] = (np.abs(rng.standard_normal(int(pos.sum()))) * 10.0 ** rng.uniform(-30, 0, int(pos.sum()))).astype(np.float32)
    rows.append(r)
    x = np.stack(rows)
    lens = np.full(x.shape[0], S, np.int32)
    got = rn.run(x, lens, K, options=rn.options(shape=shape, force_ctas_per_group=G))
    assert_matches_oracle(x, lens, got, K, label=f"far K-th S={S} K={K} shape={shape} G={G}")
    assert rn.workspace_clean()


@pytest.mark.parametrize("G", [1, 3])
def test_poison_beyond_length_is_never_used(rn, G):
    w = workloads.make("decode_batch", 8)
    x = w.logits.copy()
    cols = np.arange(x.shape[1])[None, :]
    beyond = cols >= w.lengths[:, None]
    x[beyond & (cols % 2 == 0)] = np.nan
    x[beyond & (cols % 2 == 1)] = np.inf
    got = rn.run(x, w.lengths, w.topk, options=rn.options(force_ctas_per_group=G))
    assert_matches_oracle(w.logits, w.lengths, got, w.topk, label="poison")


@pytest.mark.parametrize("shift", [1, 2, 3])
@pytest.mark.parametrize("stride_delta", [0, 1, 3])
def test_unaligned_rows(rn, shift, stride_delta):
    rng = np.random.default_rng(shift * 7 + stride_delta)
    S = 20000 + stride_delta
    x = rng.standard_normal((5, S)).astype(np.float32)
    lens = np.array([S, S - 1, 3000, 12345, 2049], np.int32)
    for G, shape in ((1, 0), (2, 0), (3, 4), (1, 5), (2, 5)):
        got = rn.run(x, lens, 2048, pad_front=shift, options=rn.options(force_ctas_per_group=G, shape=shape))
        assert_matches_oracle(x, lens, got, 2048, label=f"shift={shift} S={S} G={G} shape={shape}")


def test_lengths_are_clamped_and_flagged(rn):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 5000)).astype(np.float32)
    lens = np.array([-3, 99999, 5000, 600], np.int32)
    rn.sel.reset()
    got = rn.run(x, lens, 512, check_status=False)
    assert_matches_oracle(x, lens, got, 512, label="clamp")
    assert rn.sel.status() & rn.sar.TOPK_DEV_LENGTH_CLAMPED
    rn.sel.reset()
    assert rn.sel.status() == 0


def test_many_rows_per_cta_and_per_group(rn):
    rng = np.random.default_rng(9)
    S = 6000
    x = np.round(rng.standard_normal((300, S)) * 4).astype(np.float32) / 4
    lens = rng.integers(0, S, 300, endpoint=True).astype(np.int32)
    # 4 CTAs: 75 rows each, beyond the shared-memory length cache
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=4, force_ctas_per_group=1))
    assert_matches_oracle(x, lens, got, 1024, label="G=1 persistent")
    # the paired shape, 3 CTAs: 100 rows each
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=3, shape=2))
    assert_matches_oracle(x, lens, got, 1024, label="paired persistent")
    # the small shape, 5 CTAs: 60 rows each
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=5, shape=3))
    assert_matches_oracle(x, lens, got, 1024, label="small persistent")
    # the short-row kernel, 7 CTAs: 42 or 43 rows each (32 warps), 9 CTAs (16 warps)
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=7, shape=4))
    assert_matches_oracle(x, lens, got, 1024, label="short-row persistent")
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=9, shape=5))
    assert_matches_oracle(x, lens, got, 1024, label="short-row 16-warp persistent")
    # the wide shape on whole rows, 6 CTAs
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=6, shape=1))
    assert_matches_oracle(x, lens, got, 1024, label="wide persistent")
    # 2 groups of 4 CTAs: every group loops over 150 rows, reusing its workspace
    got = rn.run(x, lens, 1024, options=rn.options(max_ctas=8, force_ctas_per_group=4))
    assert_matches_oracle(x, lens, got, 1024, label="G=4 persistent")
    assert rn.workspace_clean()
