"""Host-side planning, checked without a GPU through ``muon_plan_workspace_size``:
orientation into (r, c) buckets, the device workspace a plan allocates, and the
chunks a workspace cap or ``chunks`` option splits the step into."""
import ctypes

import pytest

import matrix_orthogonalising_optimizer_muon_gb300 as mu

# One Qwen2.5-7B decoder layer (q, k, v, o, gate, up, down), stored as out x in.
LAYER = [(3584, 3584), (512, 3584), (512, 3584), (3584, 3584),
         (18944, 3584), (18944, 3584), (3584, 18944)]
PER_HEAD = [(128, 3584)] * 1008 + [(512, 3584)] * 28
MIXED = [(300, 1000), (1000, 300), (64, 64), (129, 4096), (4096, 256)]
BIG = (18944, 3584)


def ws(shapes, **opts):
    return mu.plan_workspace_size(shapes, **opts)


def r8(x):
    return (x + 7) // 8 * 8


def r256(x):
    return (x + 255) // 256 * 256


def held(shapes, batched_small=False):
    """Bytes the NS step must hold per matrix: the bf16 X0 (r x c, rows padded to 8)
    and, for matrices on the batched products, the seven r x r Gram-space buffers
    (G twice, P, T, Q twice, a bf16 copy of Q)."""
    t = 0
    for m, n in shapes:
        r, c = min(m, n), max(m, n)
        t += 2 * r * r8(c)
        if r > 128 or batched_small:
            t += 7 * 2 * r * r8(r)
    return t


def test_plan_sizing_needs_no_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("checks the host-only path where no GPU is present")
    lib = mu.load()
    arr = (mu.MuonShape * 1)(mu.MuonShape(*BIG))
    h = ctypes.c_void_p()
    assert lib.muon_plan_create(arr, 1, mu.MUON_BF16, None, ctypes.byref(h)) == mu.MUON_ERR_CUDA
    out = ws([BIG])
    assert out["n_buckets"] == 1 and out["n_chunks"] == 1 and out["workspace_bytes"] > 0


def test_buckets_group_oriented_shapes():
    # (m, n) and (n, m) orient to the same r x c (transpose when m > n)
    assert ws([(3584, 18944), (18944, 3584)])["n_buckets"] == 1
    assert ws([(300, 1000), (1000, 300), (1000, 301)])["n_buckets"] == 2
    # the 7B layer holds three oriented shapes: 3584 x 3584, 512 x 3584, 3584 x 18944
    assert ws(LAYER) == {"workspace_bytes": ws(LAYER)["workspace_bytes"], "n_buckets": 3, "n_chunks": 1}
    assert ws(LAYER * 28)["n_buckets"] == 3
    assert ws(PER_HEAD)["n_buckets"] == 2
    assert ws(MIXED)["n_buckets"] == 4


@pytest.mark.parametrize("shapes", [[BIG], LAYER, LAYER * 28, PER_HEAD, MIXED], ids=["big", "layer", "28l", "heads", "mixed"])
def test_workspace_holds_the_step_and_little_else(shapes):
    need = held(shapes)
    got = ws(shapes)["workspace_bytes"]
    assert got >= need
    # the rest: RowNorm's column partial sums of each stored m > n matrix (one float per
    # 64 stored rows per column), then per-matrix tables, partial sums and launch lists
    colstats = sum(4 * -(-m // 64) * n for m, n in shapes if m > n)
    assert got - need - colstats <= 0.005 * need + (1 << 20)


def test_fused_matrices_hold_no_gram_buffers():
    # r <= 128 runs on one SM per matrix with its r x r operands on chip; taking the
    # batched products instead (generic_small) adds exactly the seven r x r buffers
    k = 40
    small = [(128, 3584)] * k
    extra = ws(small, generic_small=True)["workspace_bytes"] - ws(small)["workspace_bytes"]
    assert extra == 7 * r256(k * 128 * 128 * 2)
    # a matrix with r > 128 is batched either way
    assert ws([BIG], generic_small=True) == ws([BIG])


def test_restarts_add_the_second_iterate_buffer():
    r, c = 3584, 18944
    extra = ws([BIG], max_ns_steps=10)["workspace_bytes"] - ws([BIG])["workspace_bytes"]
    assert extra == r256(r * c * 2)
    # with restarts, r <= 128 matrices leave the fused kernel for the batched path
    small = [(128, 3584)] * 8
    assert ws(small, max_ns_steps=10)["workspace_bytes"] >= held(small, batched_small=True) + 8 * 128 * 3584 * 2


@pytest.mark.parametrize("opts", [{}, {"max_ns_steps": 10}, {"generic_small": True}], ids=["plain", "restarts", "generic"])
@pytest.mark.parametrize("shapes", [[BIG], [BIG, BIG], LAYER, LAYER * 28, PER_HEAD, MIXED],
                         ids=["big", "big2", "layer", "28l", "heads", "mixed"])
def test_cap_equal_to_the_reported_size_fits_exactly(shapes, opts):
    full = ws(shapes, **opts)
    assert ws(shapes, workspace_bytes=full["workspace_bytes"], **opts) == full
    cap = full["workspace_bytes"] - 1
    if len(shapes) == 1:
        with pytest.raises(mu.MuonError) as e:
            ws(shapes, workspace_bytes=cap, **opts)
        assert e.value.code == mu.MUON_ERR_OOM
    else:
        less = ws(shapes, workspace_bytes=cap, **opts)
        assert less["n_chunks"] >= 2 and less["workspace_bytes"] <= cap


def test_smaller_caps_give_more_chunks_and_stay_within_the_cap():
    prev = 0
    for cap in (40e9, 20e9, 10e9, 5e9, 2e9, 1e9, 6e8):
        out = ws(LAYER * 28, workspace_bytes=int(cap))
        assert out["workspace_bytes"] <= cap
        assert out["n_chunks"] >= prev
        # every chunk holds each of its shapes in one bucket
        assert out["n_chunks"] <= out["n_buckets"] <= 3 * out["n_chunks"]
        prev = out["n_chunks"]
    # below the tables plus the largest single matrix there is no plan
    with pytest.raises(mu.MuonError) as e:
        ws(LAYER * 28, workspace_bytes=4 * 10 ** 8)
    assert e.value.code == mu.MUON_ERR_OOM


def test_chunks_option_splits_the_region():
    one = ws(LAYER * 28)
    prev_bytes, prev_chunks = one["workspace_bytes"], 1
    for k in (2, 4, 8, 16, 32):
        out = ws(LAYER * 28, chunks=k)
        assert out["n_chunks"] >= k and out["n_chunks"] >= prev_chunks
        assert out["workspace_bytes"] < prev_bytes
        # each chunk's region is about 1/k of the whole (or one matrix's, if larger)
        assert out["workspace_bytes"] <= one["workspace_bytes"] / k + held([BIG]) + (64 << 20)
        prev_bytes, prev_chunks = out["workspace_bytes"], out["n_chunks"]
    # never more chunks than matrices; chunks 0 and 1 mean one chunk
    assert ws(MIXED, chunks=1000)["n_chunks"] <= len(MIXED)
    assert ws(LAYER, chunks=0) == ws(LAYER, chunks=1) == ws(LAYER)


def test_sizing_rejects_what_plan_create_rejects():
    lib = mu.load()
    b, nb, nc = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    bad = (mu.MuonShape * 2)(mu.MuonShape(4, 8), mu.MuonShape(0, 3))
    f = lib.muon_plan_workspace_size
    assert f(bad, 2, mu.MUON_BF16, None, ctypes.byref(b), ctypes.byref(nb), ctypes.byref(nc)) == mu.MUON_ERR_INVALID_ARG
    assert f(bad, 0, mu.MUON_BF16, None, None, None, None) == mu.MUON_ERR_INVALID_ARG
    assert f(None, 1, mu.MUON_BF16, None, None, None, None) == mu.MUON_ERR_INVALID_ARG
    assert f(bad, 1, 7, None, None, None, None) == mu.MUON_ERR_UNSUPPORTED
    big = (mu.MuonShape * 1)(mu.MuonShape(1 << 21, 4))
    assert f(big, 1, mu.MUON_F32, None, None, None, None) == mu.MUON_ERR_UNSUPPORTED
    for o in (mu.MuonPlanOpts(chunks=-1), mu.MuonPlanOpts(workspace_bytes=-1), mu.MuonPlanOpts(max_ns_steps=101)):
        assert f(bad, 1, mu.MUON_BF16, ctypes.byref(o), None, None, None) == mu.MUON_ERR_INVALID_ARG
    # NULL outputs are allowed
    assert f(bad, 1, mu.MUON_BF16, None, None, None, None) == mu.MUON_OK


def test_size_limits():
    # each side up to 2^20, r = min(m, n) up to 32768; sizing needs no memory
    assert ws([(1 << 20, 32768), (32768, 1 << 20), (1, 1 << 20)])["n_buckets"] == 2
    for bad in ([((1 << 20) + 1, 8)], [(8, (1 << 20) + 1)], [(32769, 40000)]):
        with pytest.raises(mu.MuonError) as e:
            ws(bad)
        assert e.value.code == mu.MUON_ERR_UNSUPPORTED


def test_near_square_small_matrices_hold_no_gram_buffers():
    """Nearly square matrices with r <= 128 run in fp32 on chip (small_fp32 = 0): no r x r
    buffers, with or without generic_small; small_fp32 = -1 puts them back on the tensor
    cores (batched with generic_small: seven r x r buffers, split in two parts by
    precision 0 since they are nearly square)."""
    sq = [(96, 96)] * 4
    base = ws(sq)["workspace_bytes"]
    assert ws(sq, generic_small=True)["workspace_bytes"] == base
    rr = r256(4 * 96 * r8(96) * 2)
    extra = ws(sq, generic_small=True, small_fp32=-1)["workspace_bytes"] - base
    assert extra == 7 * r256(2 * 4 * 96 * r8(96) * 2)    # split: two parts per matrix
    extra_plain = ws(sq, generic_small=True, small_fp32=-1, precision=-1)["workspace_bytes"] - base
    assert extra_plain == 7 * rr


def test_split_precision_doubles_the_split_buffers():
    """precision 0 splits nearly square batched buckets only (r <= split_max_r): their seven
    r x r buffers hold two parts per matrix; level 2 also doubles X0."""
    sq, rect = (256, 256), (256, 1024)
    rr = r256(256 * 256 * 2)
    assert ws([sq])["workspace_bytes"] - ws([sq], precision=-1)["workspace_bytes"] == 7 * (r256(2 * rr) - rr)
    assert ws([rect])["workspace_bytes"] == ws([rect], precision=-1)["workspace_bytes"]
    assert ws([sq], split_max_r=128)["workspace_bytes"] == ws([sq], precision=-1)["workspace_bytes"]
    x = r256(256 * 1024 * 2)
    two = ws([rect], precision=2)["workspace_bytes"] - ws([rect], precision=-1)["workspace_bytes"]
    assert two == 7 * (r256(2 * rr) - rr) + x
    # the 7B layer's squares (r = 3584) and the DiT block's (r = 2048) stay plain
    assert ws(LAYER) == ws(LAYER, precision=-1)
    assert ws([(2048, 2048)]) == ws([(2048, 2048)], precision=-1)


def test_dim0_shard_plans_hold_no_newton_schulz_buffers():
    """opts.full_rows makes a RowNorm-only plan over dim-0 shards: no X0 or r x r buffers,
    and row counts above the full matrix's are refused."""
    shards = [(512, 2048), (1024, 2048), (2048, 512)]
    plain = ws(shards)["workspace_bytes"]
    sharded = ws(shards, full_rows=[6144, 2048, 4096])["workspace_bytes"]
    assert sharded < plain and sharded < 4 << 20
    with pytest.raises(mu.MuonError):
        ws(shards, full_rows=[256, 2048, 4096])   # a shard of 512 rows of a 256-row matrix


def test_precision_of_splits_buckets_per_matrix():
    """opts.precision_of: matrices of one oriented shape with different levels form separate
    buckets, each sized for its own level."""
    sq = [(256, 256)] * 2
    assert ws(sq, precision_of=[-1, 1])["n_buckets"] == 2
    assert ws(sq, precision_of=[1, 1])["n_buckets"] == 1
    rr = r256(256 * 256 * 2)   # one plain r x r buffer of one matrix
    plain2 = ws(sq, precision_of=[-1, -1])["workspace_bytes"]
    mixed = ws(sq, precision_of=[-1, 1])["workspace_bytes"]
    assert mixed - plain2 == 7 * rr                  # the split matrix's seven buffers hold two parts
    assert ws(sq, precision_of=[0, 0]) == ws(sq)     # 0: the plan-wide rule
