"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every test compares element by element on seeded inputs, within
|err| <= 1e-2 * sum_k |a_ik b_kj| (+ 1e-2 |bias_j|) + 1e-5, and also checks the
tight diagnostic that catches dropped or repeated K-slices.  Where the exact
result is an integer below 2^24 the comparison is bitwise.
"""
import numpy as np
import pytest
import torch

import grouped_gemm_persistent_gb300 as tg
import oracle
from grouped_gemm_persistent_gb300 import workloads as wl

from parity import check_dense, oracle_dense, run_dense, sample_rows, to_device, to_f64

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]   # (A column-major, B column-major)


def pad8(x: int) -> int:
    """Leading dimensions are padded to 8 bf16 elements (TMA: row strides are multiples of 16 bytes)."""
    return -(-x // 8) * 8


def lds(M, N, K, a_col, b_col):
    return dict(lda=pad8(M if a_col else K), ldb=pad8(K if b_col else N))


TILES = ["1x128", "1x256", "2x128", "2x256"]   # <cta_group>x<BN>: single CTA or CTA pair, tile width


@pytest.fixture(params=TILES)
def tile(request, monkeypatch):
    """Force one kernel variant (the library reads TG_TILE at every call)."""
    monkeypatch.setenv("TG_TILE", request.param)
    return request.param


@pytest.fixture(autouse=True, scope="module")
def _built():
    from grouped_gemm_persistent_gb300.build import build
    build()
    tg.load()


def _sync_ok():
    tg.device_status()


# ------------------------------------------------------------------------------------------ dense

def test_dense_256_workload():
    case = wl.dense_case("dense_256")
    c = run_dense(case)
    _sync_ok()
    check_dense(case, c)


@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("epi", ["none", "bias", "bias_gelu"])
@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
def test_dense_ragged_all_variants(a_col, b_col, epi, c_dtype, tile):
    # spans several tiles with a ragged tail in M, N and K (K not a multiple of 64)
    case = wl.dense_random(333, 392, 200, seed=100, dist="uniform", a_col_major=a_col, b_col_major=b_col,
                           epi=epi, c_dtype=c_dtype, **lds(333, 392, 200, a_col, b_col))
    c = run_dense(case)
    _sync_ok()
    check_dense(case, c)


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (1, 8, 8), (129, 264, 65), (512, 256, 1024), (17, 16, 3000),
                                   (640, 136, 128), (7, 520, 72)])
@pytest.mark.parametrize("a_col,b_col", [(False, False), (False, True)])
def test_dense_shapes(M, N, K, a_col, b_col, tile):
    case = wl.dense_random(M, N, K, seed=M * 7 + N * 3 + K, dist="normal", a_col_major=a_col, b_col_major=b_col,
                           epi="bias", c_dtype="bf16", **lds(M, N, K, a_col, b_col))
    c = run_dense(case)
    _sync_ok()
    check_dense(case, c)


def test_padded_leading_dimensions():
    case = wl.dense_random(200, 136, 150, seed=9, dist="normal", lda=160, ldb=144, epi="bias_gelu")
    c_full = torch.full((200, 152), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = c_full[:, :136]
    run_dense(case, out)
    _sync_ok()
    check_dense(case, out)
    assert torch.isnan(c_full[:, 136:].float()).all(), "columns beyond N were written"


def test_integer_exact_bitwise(tile):
    # integers in [-4, 4]: every fp32 partial sum is exact, so C must equal the
    # exact result bit for bit (fp32 out) and its RNE rounding (bf16 out)
    for a_col, b_col in LAYOUTS:
        case = wl.dense_random(300, 264, 640, seed=5, dist="int4", a_col_major=a_col, b_col_major=b_col,
                               c_dtype="f32", **lds(300, 264, 640, a_col, b_col))
        y, _ = oracle_dense(case)
        c = run_dense(case)
        _sync_ok()
        assert np.array_equal(to_f64(c), y), f"fp32 output not exact for layouts {a_col, b_col}"
        case.c_dtype = "bf16"
        c16 = run_dense(case)
        _sync_ok()
        want = torch.from_numpy(y).to(torch.bfloat16)
        assert torch.equal(c16.cpu().view(torch.int16), want.view(torch.int16))


def test_identity_and_permutation_exact(tile):
    M, N = 256, 192
    rng = np.random.default_rng(1)
    perm = rng.permutation(M)
    P = torch.zeros((M, M), dtype=torch.bfloat16)
    P[torch.arange(M), torch.from_numpy(perm)] = 1
    B = torch.randn((M, N), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    c = tg.gemm(P.cuda(), B.cuda(), out_dtype=torch.float32)
    _sync_ok()
    assert torch.equal(c.cpu(), B.float()[torch.from_numpy(perm)])
    # B = I: C = A; column-major B view
    A = torch.randn((M, 128), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    eye = torch.eye(128, dtype=torch.bfloat16).cuda()
    c = tg.gemm(A.cuda(), eye.t().contiguous().t(), out_dtype=torch.float32)
    _sync_ok()
    assert torch.equal(c.cpu(), A.float())


def test_k_zero_is_epilogue_of_zero(tile):
    M, N = 130, 200
    bias = (torch.randn(N, generator=torch.Generator().manual_seed(4)) * 3).to(torch.bfloat16)
    a = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    for epi in ("none", "bias", "bias_gelu"):
        c = tg.gemm(a, b, bias=bias.cuda(), epilogue=epi, out_dtype=torch.float32)
        _sync_ok()
        z = torch.zeros((M, N), dtype=torch.float64) + (bias.double() if epi != "none" else 0)
        want = torch.nn.functional.gelu(z, approximate="tanh") if epi == "bias_gelu" else z
        assert torch.allclose(c.cpu().double(), want, rtol=2e-3, atol=1e-5), epi


def test_empty_m_or_n_writes_nothing():
    a = torch.randn((0, 64), device="cuda").to(torch.bfloat16)
    b = torch.randn((64, 64), device="cuda").to(torch.bfloat16)
    out = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    tg.gemm(a, b, out)
    _sync_ok()


def test_guard_bands_untouched(tile):
    case = wl.dense_random(300, 264, 128, seed=12, dist="normal", epi="bias")
    big = torch.full((300 + 64, 264 + 40), float("inf"), dtype=torch.float32, device="cuda")
    out = big[32:332, 8:272]
    run_dense(wl.dense_random(300, 264, 128, seed=12, dist="normal", epi="bias", c_dtype="f32"), out)
    _sync_ok()
    case.c_dtype = "f32"
    check_dense(case, out)
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[32:332, 8:272] = False
    assert torch.isinf(big[mask]).all(), "a write landed outside C"


def test_deterministic_bitwise(tile):
    case = wl.dense_random(1000, 1000, 1000, seed=13, dist="normal", epi="bias_gelu")
    c1 = run_dense(case)
    c2 = run_dense(case)
    _sync_ok()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_nan_stays_in_its_row():
    case = wl.dense_random(256, 256, 256, seed=14, dist="normal", c_dtype="f32")
    case.a = case.a.clone()
    case.a[37, 11] = float("nan")
    c = run_dense(case).cpu()
    _sync_ok()
    assert torch.isnan(c[37]).all()
    rest = torch.cat([c[:37], c[38:]])
    assert torch.isfinite(rest).all()


def test_side_stream():
    case = wl.dense_random(512, 512, 512, seed=15, dist="normal")
    a, b = case.a.cuda(), case.b.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = tg.gemm(a, b, stream=s)
    tg.device_status(s)
    check_dense(case, c)


# ------------------------------------------------------------------------------------------ fp16 operands

def _f16_case(M, N, K, seed, a_col, b_col, scale=0.25, ints=False):
    gen = torch.Generator().manual_seed(seed)
    def draw(shape):
        if ints:
            return torch.randint(-4, 5, shape, generator=gen).to(torch.float16)
        return (torch.randn(shape, generator=gen) * scale).to(torch.float16)
    a = draw((K, M) if a_col else (M, K))
    b = draw((N, K) if b_col else (K, N))
    bias = (torch.randn(N, generator=gen) * 0.1).to(torch.float16)
    return a, b, bias


@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_f16_operands(a_col, b_col, epi, out_dtype, tile):
    M, N, K = 264, 392, 200
    a, b, bias = _f16_case(M, N, K, 61, a_col, b_col)
    da, db = a.cuda(), b.cuda()
    out = tg.gemm(da.t() if a_col else da, db.t() if b_col else db, bias=bias.cuda(), epilogue=epi, out_dtype=out_dtype)
    _sync_ok()
    h = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    y, s = oracle.gemm(h(a), h(b), a_col_major=a_col, b_col_major=b_col, bias=h(bias), epi=epi, in_dtype="f16")
    r = oracle.compare(to_f64(out), y, s, np.abs(bias.double().numpy()) if epi != "none" else None)
    assert r["ok"] and r["max_tight"] < 4.0, r


def test_f16_integer_exact(tile):
    a, b, _ = _f16_case(300, 264, 640, 62, False, True, ints=True)
    out = tg.gemm(a.cuda(), b.cuda().t(), out_dtype=torch.float32)
    _sync_ok()
    exact = (a.double() @ b.double().t()).numpy()
    assert np.array_equal(to_f64(out), exact)
    out16 = tg.gemm(a.cuda(), b.cuda().t(), out_dtype=torch.float16)
    _sync_ok()
    assert torch.equal(out16.cpu().view(torch.int16), torch.from_numpy(exact).to(torch.float16).view(torch.int16))


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.float32])
def test_f16_wide_b_view_integer_exact(out_dtype, tile):
    # fp16 operands with N-major B and N % 64 == 0 (the 64-column-chunk view of B), a
    # partial last N-tile and a ragged K: integer inputs, so the result is exact
    a, b, _ = _f16_case(333, 320, 200, 64, False, False, ints=True)
    out = tg.gemm(a.cuda(), b.cuda(), out_dtype=out_dtype)
    _sync_ok()
    exact = (a.double() @ b.double()).numpy()
    if out_dtype == torch.float32:
        assert np.array_equal(to_f64(out), exact)
    else:
        assert torch.equal(out.cpu().view(torch.int16), torch.from_numpy(exact).to(torch.float16).view(torch.int16))


def test_grouped_mixed_bf16_and_f16_problems(tile):
    gen = torch.Generator().manual_seed(63)
    keep, probs, refs = [], [], []
    for M, N, K, dt in [(100, 136, 64, torch.float16), (257, 264, 200, torch.bfloat16), (64, 136, 128, torch.float16)]:
        a = (torch.randn((M, K), generator=gen) / 4).to(dt)
        b = (torch.randn((K, N), generator=gen) / 4).to(dt)
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        da, db = a.cuda(), b.cuda()
        keep += [da, db, out]
        probs.append(tg.make_problem(da, db, out))
        refs.append((a, b, out, "f16" if dt == torch.float16 else "bf16"))
    tg.grouped_gemm_table(probs)
    _sync_ok()
    for a, b, out, ind in refs:
        h = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        y, s = oracle.gemm(h(a), h(b), in_dtype=ind)
        r = oracle.compare(to_f64(out), y, s)
        assert r["ok"] and r["max_tight"] < 4.0, r


# ------------------------------------------------------------------------------------------ in-kernel broadcast

@pytest.mark.parametrize("U,repeat,N,K", [(37, 5, 136, 72), (300, 1, 264, 128), (5, 300, 128, 64),
                                          (129, 3, 392, 200), (256, 40, 128, 1024)])
@pytest.mark.parametrize("epi", ["none", "bias", "bias_gelu"])
def test_bcast_matches_materialised(U, repeat, N, K, epi):
    gen = torch.Generator().manual_seed(U + repeat + N + K)
    users = (torch.randn((U, K), generator=gen) / 4).to(torch.bfloat16)
    b = (torch.randn((K, N), generator=gen) / 4).to(torch.bfloat16)
    bias = (torch.randn(N, generator=gen) * 0.1).to(torch.bfloat16)
    out = torch.full((U * repeat, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    tg.gemm_bcast(users.cuda(), b.cuda(), repeat, out, bias=bias.cuda(), epilogue=epi)
    _sync_ok()
    a = users.repeat_interleave(repeat, dim=0)          # the materialised A the definition refers to
    y, s = oracle.gemm(wl.bf16_bits(a), wl.bf16_bits(b), bias=wl.bf16_bits(bias), epi=epi)
    r = oracle.compare(to_f64(out), y, s, np.abs(bias.double().numpy()) if epi != "none" else None)
    assert r["ok"] and r["max_tight"] < 4.0, r


def test_bcast_equals_dense_on_materialised_bitwise(monkeypatch):
    monkeypatch.setenv("TG_STREAM_K", "0")    # same summation order on both paths
    case = wl.dense_case("skinny_bcast")
    dense = run_dense(case)
    bc = tg.gemm_bcast(case.users.cuda(), case.b.cuda(), case.repeat, bias=case.bias.cuda(), epilogue="bias")
    _sync_ok()
    assert torch.equal(dense.view(torch.int16), bc.view(torch.int16))


def test_workload_skinny_bcast_in_kernel_broadcast_full():
    case = wl.dense_case("skinny_bcast")
    c = tg.gemm_bcast(case.users.cuda(), case.b.cuda(), case.repeat, bias=case.bias.cuda(), epilogue="bias")
    _sync_ok()
    check_dense(case, c)


# ------------------------------------------------------------------------------------------ grouped

def _grouped_problems(counts, N, K, seed, epi="none", c_dtype="bf16", b_col=False):
    case = wl.grouped_random(counts, N, K, seed, epi=epi, c_dtype=c_dtype)
    a = case.a.cuda()
    bst = case.b if not b_col else case.b.transpose(1, 2).contiguous()   # [G, N, K] storage if col-major
    b = bst.cuda()
    dt = torch.float32 if c_dtype == "f32" else torch.bfloat16
    out = torch.empty((int(np.sum(counts)), N), dtype=dt, device="cuda")
    bias = case.bias.cuda() if case.bias is not None else None
    return case, a, b, out, bias


def _check_grouped(case, out, b_col=False, rows_per_group=None):
    c_all = out.float().cpu().double().numpy()
    for g in range(case.G):
        r0, r1 = case.offsets[g], case.offsets[g + 1]
        if r1 == r0:
            continue
        a_g = wl.bf16_bits(case.a[r0:r1])
        b_g = wl.bf16_bits(case.b[g] if not b_col else case.b[g].t().contiguous())
        bias = wl.bf16_bits(case.bias[g]) if case.bias is not None else None
        rows = None if rows_per_group is None else rows_per_group[g]
        y, s = oracle.gemm(a_g, b_g, b_col_major=b_col, bias=bias, epi=case.epi, rows=rows)
        c = c_all[r0:r1] if rows is None else c_all[r0 + rows]
        bias_abs = np.abs(case.bias[g].double().numpy()) if case.bias is not None else None
        r = oracle.compare(c, y, s, bias_abs)
        assert r["ok"] and r["max_tight"] < 4.0, f"group {g}: {r}"


@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
@pytest.mark.parametrize("b_col", [False, True])
def test_grouped_ragged_with_empty_groups(epi, b_col, tile):
    counts = [0, 300, 5, 0, 130, 257, 1, 0]        # empty first, middle and last
    case, a, b, out, bias = _grouped_problems(counts, 136, 200, 21, epi=epi, b_col=b_col)
    sentinel = torch.full_like(out, float("nan"))
    out.copy_(sentinel)
    bview = b.transpose(1, 2) if b_col else b      # logical [G, K, N]
    tg.moe_grouped_gemm(a, bview, counts, out, bias=bias, epilogue=epi)
    _sync_ok()
    assert not torch.isnan(out.float()).any(), "a row of a non-empty group was not written"
    _check_grouped(case, out, b_col=b_col)


def test_grouped_more_problems_than_the_shared_table():
    # The kernel keeps each problem's first tile in shared memory for up to 382
    # problems and walks the problem array in global memory beyond that: 420
    # non-empty problems (and a few empty ones) take the global walk.
    rng = np.random.default_rng(31)
    counts = [int(c) for c in rng.integers(1, 40, size=424)]
    for i in (0, 100, 250, 423):
        counts[i] = 0
    case, a, b, out, bias = _grouped_problems(counts, 64, 64, 32, epi="bias")
    sentinel = torch.full_like(out, float("nan"))
    out.copy_(sentinel)
    tg.moe_grouped_gemm(a, b, counts, out, bias=bias, epilogue="bias")
    _sync_ok()
    assert not torch.isnan(out.float()).any(), "a row of a non-empty group was not written"
    _check_grouped(case, out)


def test_grouped_single_group_matches_dense_bitwise(tile, monkeypatch):
    monkeypatch.setenv("TG_STREAM_K", "0")    # same summation order on both paths
    case = wl.dense_random(700, 392, 320, seed=22, dist="normal", epi="bias")
    a, b, bias = case.a.cuda(), case.b.cuda(), case.bias.cuda()
    dense = tg.gemm(a, b, bias=bias, epilogue="bias")
    grouped = tg.moe_grouped_gemm(a, b[None], [700], bias=bias[None], epilogue="bias")
    _sync_ok()
    assert torch.equal(dense.view(torch.int16), grouped.view(torch.int16))


def test_grouped_mixed_layouts_and_dtypes(tile):
    # problems of different layouts and output types in one call (one launch per class)
    gen = torch.Generator().manual_seed(23)
    probs, refs = [], []
    specs = [(100, 136, 64, False, False, "bf16"), (260, 128, 200, False, True, "f32"),
             (0, 128, 64, False, False, "bf16"), (40, 264, 72, True, False, "bf16"),
             (129, 136, 128, False, False, "f32")]
    keep = []
    for (M, N, K, a_col, b_col, cd) in specs:
        a = (torch.randn((K, M) if a_col else (M, K), generator=gen) / 8).to(torch.bfloat16)
        b = (torch.randn((N, K) if b_col else (K, N), generator=gen) / 8).to(torch.bfloat16)
        da, db = a.cuda(), b.cuda()
        out = torch.empty((M, N), dtype=torch.float32 if cd == "f32" else torch.bfloat16, device="cuda")
        keep += [da, db, out]
        probs.append(tg.make_problem(da.t() if a_col else da, db.t() if b_col else db, out))
        refs.append((a, b, a_col, b_col, out))
    tg.grouped_gemm_table(probs)
    _sync_ok()
    for a, b, a_col, b_col, out in refs:
        if out.shape[0] == 0:
            continue
        y, s = oracle.gemm(wl.bf16_bits(a), wl.bf16_bits(b), a_col_major=a_col, b_col_major=b_col)
        r = oracle.compare(to_f64(out), y, s)
        assert r["ok"] and r["max_tight"] < 4.0, r


# Half tiles: with CTA pairs, a problem's last M-tile with at most 128 rows left runs
# as M = 128 MMAs (64 rows per CTA, accumulator columns split over the TMEM lane
# halves).  Row counts around every boundary, both tile widths, all layouts.
HALF_COUNTS = [1, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 300, 384, 385, 640]


@pytest.mark.parametrize("tile_shape", ["2x256", "2x128"])
@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
def test_grouped_half_tiles(tile_shape, a_col, b_col, c_dtype, monkeypatch):
    monkeypatch.setenv("TG_TILE", tile_shape)
    gen = torch.Generator().manual_seed(61)
    N, K = 264, 136
    probs, refs, keep = [], [], []
    for M in HALF_COUNTS:
        a = (torch.randn((K, M) if a_col else (M, K), generator=gen) / 8).to(torch.bfloat16)
        b = (torch.randn((N, K) if b_col else (K, N), generator=gen) / 8).to(torch.bfloat16)
        bias = (torch.randn((N,), generator=gen) / 10).to(torch.bfloat16)
        if a_col:
            a = torch.nn.functional.pad(a, (0, (-M) % 8))[:, :M]      # column stride a multiple of 8
        da, db, dbias = to_device(a), b.cuda(), bias.cuda()
        out = torch.full((M, N), float("nan"), dtype=torch.float32 if c_dtype == "f32" else torch.bfloat16,
                         device="cuda")
        keep += [da, db, dbias, out]
        probs.append(tg.make_problem(da.t() if a_col else da, db.t() if b_col else db, out, bias=dbias,
                                     epilogue="bias_gelu"))
        refs.append((a, b, bias, out))
    tg.grouped_gemm_table(probs)
    _sync_ok()
    for a, b, bias, out in refs:
        y, s = oracle.gemm(wl.bf16_bits(a.contiguous()), wl.bf16_bits(b), a_col_major=a_col, b_col_major=b_col,
                           bias=wl.bf16_bits(bias), epi="bias_gelu")
        r = oracle.compare(to_f64(out), y, s, np.abs(bias.double().numpy()))
        assert r["ok"] and r["max_tight"] < 4.0, (out.shape, r)


@pytest.mark.parametrize("tile_shape", ["2x256", "2x128"])
def test_moe_half_tiles_device_counts(tile_shape, monkeypatch):
    monkeypatch.setenv("TG_TILE", tile_shape)
    counts = [129, 1, 128, 0, 64, 257, 385, 127]
    case, a, b, bias, T = _moe_case(counts, 200, 136, 62, epi="bias_gelu", extra_rows=40)
    out = torch.full((T, 200), float("nan"), dtype=torch.bfloat16, device="cuda")
    tg.moe_gemm_device(a, b, torch.tensor(counts, dtype=torch.int32, device="cuda"), out, bias=bias,
                       epilogue="bias_gelu")
    _sync_ok()
    total = int(np.sum(counts))
    assert torch.isnan(out[total:].float()).all(), "rows past the counts were written"
    _check_grouped(case, out[:total])


# ------------------------------------------------------------------------------------------ MoE, device counts

def _moe_case(counts, N, K, seed, epi="none", b_col=False, extra_rows=0):
    case = wl.grouped_random(counts, N, K, seed, epi=epi)
    T = int(np.sum(counts)) + extra_rows
    a = torch.zeros((T, K), dtype=torch.bfloat16)
    a[: case.a.shape[0]] = case.a
    a = a.cuda()
    bst = case.b if not b_col else case.b.transpose(1, 2).contiguous()
    b = bst.cuda()
    bview = b.transpose(1, 2) if b_col else b
    bias = case.bias.cuda() if case.bias is not None else None
    return case, a, bview, bias, T


@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
@pytest.mark.parametrize("b_col", [False, True])
@pytest.mark.parametrize("c_dtype", [torch.bfloat16, torch.float32])
def test_moe_device_counts_equal_grouped_bitwise(epi, b_col, c_dtype, tile):
    counts = [0, 300, 5, 0, 130, 257, 1, 0, 64]
    case, a, b, bias, T = _moe_case(counts, 136, 200, 51, epi=epi, b_col=b_col)
    dev = torch.tensor(counts, dtype=torch.int32, device="cuda")
    out_dev = torch.full((T, 136), float("nan"), dtype=c_dtype, device="cuda")
    tg.moe_gemm_device(a, b, dev, out_dev, bias=bias, epilogue=epi)
    out_tab = torch.empty_like(out_dev)
    tg.moe_grouped_gemm(a, b, counts, out_tab, bias=bias, epilogue=epi)
    _sync_ok()
    assert torch.equal(out_dev.view(torch.int16 if c_dtype != torch.float32 else torch.int32),
                       out_tab.view(torch.int16 if c_dtype != torch.float32 else torch.int32))
    _check_grouped(case, out_dev, b_col=b_col)


def test_moe_rows_past_the_counts_are_untouched(tile):
    counts = [129, 0, 70]
    case, a, b, bias, T = _moe_case(counts, 264, 128, 52, extra_rows=77)
    dev = torch.tensor(counts, dtype=torch.int32, device="cuda")
    out = torch.full((T, 264), float("nan"), dtype=torch.bfloat16, device="cuda")
    tg.moe_gemm_device(a, b, dev, out)
    _sync_ok()
    used = int(sum(counts))
    assert not torch.isnan(out[:used].float()).any()
    assert torch.isnan(out[used:].float()).all(), "rows past sum(counts) were written"
    _check_grouped(case, out[:used])


def test_moe_invalid_device_counts_are_reported():
    counts_ok = [100, 50]
    case, a, b, bias, T = _moe_case(counts_ok, 136, 64, 53)
    out = torch.zeros((T, 136), dtype=torch.bfloat16, device="cuda")
    for bad in ([100, -1], [100, 51]):            # negative; sum above T
        tg.moe_gemm_device(a, b, torch.tensor(bad, dtype=torch.int32, device="cuda"), out)
        with pytest.raises(tg.TGError) as ei:
            tg.device_status()
        assert ei.value.status == tg.TG_ERR_INVALID_ARG
    tg.moe_gemm_device(a, b, torch.tensor(counts_ok, dtype=torch.int32, device="cuda"), out)
    _sync_ok()
    _check_grouped(case, out)


def test_workload_grouped_moe_device_counts_bitwise():
    case = wl.grouped_case("grouped_moe")
    a, b = case.a.cuda(), case.b.cuda()
    out_dev = tg.moe_gemm_device(a, b, torch.tensor(case.counts, dtype=torch.int32, device="cuda"))
    out_tab = tg.moe_grouped_gemm(a, b, case.counts)
    _sync_ok()
    assert torch.equal(out_dev.view(torch.int16), out_tab.view(torch.int16))


# ------------------------------------------------------------------------------------------ failure path

# Block 0's first work item at 256 x 256 x 4096 is a stream-K range of k-blocks
# [0, 8) in every variant; a single CTA's block 1 has [8, 16), a pair's block 1
# shares block 0's.  Withholding k-block 3 or 5 leaves the later stages of the
# ring loaded when the wait runs out; withholding in a pair's second CTA leaves
# a phase that the first CTA loaded but its partner did not, which the abort
# path closes before it waits for the loads that were issued.
@pytest.mark.parametrize("block,kb", [(0, 3), (0, 5), (1, 5)])
def test_bounded_wait_reports_timeout_and_context_survives(tile, block, kb):
    case = wl.dense_random(256, 256, 4096, seed=30, dist="normal")
    a, b = case.a.cuda(), case.b.cuda()
    if block == 1 and tile.startswith("1x"):
        kb += 8
    tg.set_wait_budget_ms(100)
    try:
        tg.debug_withhold_stage(kb, block=block)
        tg.gemm(a, b)
        with pytest.raises(tg.TGError) as ei:
            tg.device_status()
        assert ei.value.status == tg.TG_ERR_TIMEOUT
        assert "role=" in str(ei.value)
        assert "; 0 abort-path drains ran out" in str(ei.value), str(ei.value)
    finally:
        tg.set_wait_budget_ms(0)
    # nothing else was recorded after the timeout (the drain of the issued loads finished in time)
    tg.device_status()
    # the context is still usable and the record was cleared
    c = run_dense(case)
    _sync_ok()
    check_dense(case, c)


# ------------------------------------------------------------------------------------------ timeline trace

def test_timeline_trace_records_every_tile(tile):
    case = wl.dense_random(1000, 1000, 512, seed=31, dist="normal")
    a, b = case.a.cuda(), case.b.cuda()
    tiles = torch.zeros((4096, 4), dtype=torch.int64, device="cuda")
    ctas = torch.zeros((1024, 4), dtype=torch.int64, device="cuda")
    tg.debug_trace(tiles, ctas)
    c = tg.gemm(a, b)
    _sync_ok()
    check_dense(case, c)
    tr = tiles.cpu().numpy()
    used = tr[:, 1] > 0
    n = int(used.sum())
    assert n > 0 and not used[2048:].any()
    t = tr[used]
    assert (t[:, 1] <= t[:, 2]).all() and (t[:, 2] <= t[:, 3]).all()
    cr = ctas.cpu().numpy()
    live = cr[:, 0] > 0
    assert live.any()
    # {entry, set-up done, teardown start, exit} in order for every block that ran
    assert (cr[live, 0] <= cr[live, 1]).all() and (cr[live, 1] <= cr[live, 2]).all()
    assert (cr[live, 2] <= cr[live, 3]).all()
    assert set(t[:, 0].tolist()) <= set(np.flatnonzero(live).tolist())
    # slot i * U + u holds the i-th item of unit u: a unit's items run in slot order
    U = int(live.sum()) // (2 if tile.startswith("2x") else 1)
    for u in range(U):
        mine = tr[u::U]
        mine = mine[mine[:, 1] > 0]
        assert (np.diff(mine[:, 1]) > 0).all(), "a unit's work items start in slot order"
    # the trace disarms itself: a second launch leaves a fresh buffer untouched
    tiles2 = torch.zeros_like(tiles)
    tg.gemm(a, b)
    _sync_ok()
    assert not tiles2.any()


# ------------------------------------------------------------------------------------------ stream-K
# A dense launch whose tiles do not divide evenly over the resident CTAs (pairs)
# balances the tiles of its last, partial wave.  Tiles of at most 96 k-blocks
# and 256 columns run as column halves when there is room for them (next
# section); otherwise, and always under TG_STREAM_K=1 as here, as stream-K
# pieces: their k-blocks are cut into equal ranges, one per unit, run after the
# unit's first whole tile; the last piece of a tile to arrive adds the fp32
# partials in k order.
# Shapes below: (a) more tiles than resident pairs, with a small remainder
# (2304^2 x 2048: 81 pair tiles on 76 pairs, 5 tiles in 10 pieces); (b) fewer
# tiles than CTAs (512^2 x 2048: 8 tiles in 64 pieces); (c) a ragged tail in M,
# N and K; (d) two pieces per tile after a full wave (4096^2 x 2048 with B
# column-major, the 4096^3 workload's layout and plan: 28 tiles in 56 pieces).

SPLIT_SHAPES = [(2304, 2304, 2048), (512, 512, 2048), (1000, 776, 1480), (4096, 4096, 2048)]


@pytest.fixture
def stream_k(monkeypatch):
    monkeypatch.setenv("TG_STREAM_K", "1")


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
@pytest.mark.parametrize("epi", ["none", "bias_gelu"])
def test_stream_k_matches_oracle(M, N, K, epi, stream_k):
    case = wl.dense_random(M, N, K, seed=41, dist="normal", epi=epi, b_col_major=(M == 4096))
    c = run_dense(case)
    _sync_ok()
    if M * N > 4_000_000:
        check_dense(case, c, rows=sample_rows(M, 256, 160, seed=5))
    else:
        check_dense(case, c)


@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
def test_stream_k_deterministic_and_close_to_whole_tiles(c_dtype, stream_k, monkeypatch):
    case = wl.dense_random(2304, 2304, 2048, seed=42, dist="normal", c_dtype=c_dtype, epi="bias")
    c1 = run_dense(case)
    c2 = run_dense(case)
    monkeypatch.setenv("TG_STREAM_K", "0")
    c0 = run_dense(case)
    _sync_ok()
    assert torch.equal(c1, c2), "stream-K tiles must not depend on which piece finishes last"
    check_dense(case, c0)
    check_dense(case, c1)


def test_stream_k_integer_exact_bitwise(stream_k):
    # integer partial sums are exact in fp32, so the stream-K result equals the exact one
    for M, N, K in SPLIT_SHAPES[:3]:
        case = wl.dense_random(M, N, K, seed=43, dist="int4", c_dtype="f32", **lds(M, N, K, False, False))
        y, _ = oracle_dense(case)
        c = run_dense(case)
        _sync_ok()
        assert np.array_equal(to_f64(c), y), (M, N, K)


@pytest.mark.parametrize("tile_shape", TILES)
def test_stream_k_every_variant(tile_shape, stream_k, monkeypatch):
    # 640x520x1536: fewer tiles than CTAs; 2304^2 x 2048: one or two full waves and a remainder
    monkeypatch.setenv("TG_TILE", tile_shape)
    for M, N, K in [(640, 520, 1536), (2304, 2304, 2048)]:
        for a_col, b_col in LAYOUTS:
            case = wl.dense_random(M, N, K, seed=44, dist="uniform", a_col_major=a_col, b_col_major=b_col,
                                   epi="bias", **lds(M, N, K, a_col, b_col))
            c = run_dense(case)
            _sync_ok()
            check_dense(case, c)


def test_stream_k_after_full_waves_integer_exact(stream_k):
    # two pieces per tile between whole tiles (the 4096^3 workload's plan at K = 2048):
    # deterministic and integer-exact, f32 and bf16 output
    for c_dtype in ("f32", "bf16"):
        case = wl.dense_random(4096, 4096, 2048, seed=45, dist="int4", c_dtype=c_dtype, b_col_major=True)
        rows = sample_rows(4096, 256, 64, seed=6)
        y, _ = oracle_dense(case, rows=rows)
        c1 = run_dense(case)
        c2 = run_dense(case)
        _sync_ok()
        assert torch.equal(c1, c2)
        got = to_f64(c1[torch.as_tensor(rows, device=c1.device)])
        if c_dtype == "f32":
            assert np.array_equal(got, y)
        else:
            assert np.array_equal(got, to_f64(torch.from_numpy(y).to(torch.bfloat16)))


# ------------------------------------------------------------------------------------------ column halves
# With 256-wide tiles of at most 96 k-blocks and room for twice the last wave's
# tiles, each of those tiles runs as two 128-column units (N = 128 MMAs; B
# column-major through a second tensor map whose box covers half the N rows,
# B row-major through half of the 64-column boxes).  No partial sums: every
# element is one unit's fp32 accumulation in k order, so the result is bitwise
# equal to the whole-tile one.  Shapes: 2304^2 (81 pair tiles: 5 in halves);
# 4096^2 (256 pair tiles: 28 in halves, the 4096^3 workload's plan); a ragged
# 2500 x 2296 (90 tiles: 14 in halves, partial last rows and columns).

HALF_SHAPES = [(2304, 2304, 1024), (4096, 4096, 1024), (2500, 2296, 1000)]


@pytest.mark.parametrize("M,N,K", HALF_SHAPES)
@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
def test_column_halves_match_oracle_and_whole_tiles(M, N, K, a_col, b_col, monkeypatch):
    case = wl.dense_random(M, N, K, seed=46, dist="normal", a_col_major=a_col, b_col_major=b_col, epi="bias_gelu",
                           **lds(M, N, K, a_col, b_col))
    c_half = run_dense(case)
    monkeypatch.setenv("TG_STREAM_K", "0")
    c_whole = run_dense(case)
    _sync_ok()
    assert torch.equal(c_half.view(torch.int16), c_whole.view(torch.int16)), "halves differ from whole tiles"
    check_dense(case, c_half, rows=sample_rows(M, 256, 96, seed=7) if M * N > 4_000_000 else None)


def test_column_halves_integer_exact_and_guard_bands():
    M, N, K = 2304, 2304, 1024
    case = wl.dense_random(M, N, K, seed=47, dist="int4", c_dtype="f32", b_col_major=True)
    y, _ = oracle_dense(case)
    big = torch.full((M + 16, N + 24), float("inf"), dtype=torch.float32, device="cuda")
    out = big[8:8 + M, 8:8 + N]
    run_dense(case, out)
    _sync_ok()
    assert np.array_equal(to_f64(out), y)
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[8:8 + M, 8:8 + N] = False
    assert torch.isinf(big[mask]).all(), "a write landed outside C"


# ------------------------------------------------------------------------------------------ N-major B, wide view
# N-major B with N % 64 == 0 is read through the view {64 columns, k, 64-column chunk}: one
# TMA box per k-block for a CTA's share of the tile.  Chunks past N (a partial last
# N-tile, or a CTA whose whole share lies past N) read as zeros.

WIDE_SHAPES = [(333, 320, 200), (300, 640, 136), (257, 64, 520)]


@pytest.mark.parametrize("M,N,K", WIDE_SHAPES)
@pytest.mark.parametrize("a_col", [False, True])
def test_wide_b_view_integer_exact(M, N, K, a_col, tile):
    case = wl.dense_random(M, N, K, seed=M + N + K, dist="int4", a_col_major=a_col, b_col_major=False,
                           c_dtype="f32", **lds(M, N, K, a_col, False))
    y, _ = oracle_dense(case)
    c = run_dense(case)
    _sync_ok()
    assert np.array_equal(to_f64(c), y)


@pytest.mark.parametrize("epi,c_dtype", [("bias_gelu", "bf16"), ("none", "f32")])
def test_wide_b_view_equals_plain_boxes_bitwise(epi, c_dtype, tile):
    # N = 320 takes the wide view, N = 328 (not a multiple of 64) the 64-column boxes of the
    # plain map; on the same A, B columns and bias the first 320 columns agree bit for bit
    M, K, N = 333, 200, 328
    case = wl.dense_random(M, N, K, seed=48, dist="normal", epi=epi, c_dtype=c_dtype)
    a, b, bias = to_device(case.a), to_device(case.b), to_device(case.bias) if case.bias is not None else None
    dt = torch.float32 if c_dtype == "f32" else torch.bfloat16
    wide = torch.empty((M, 320), dtype=dt, device="cuda")
    plain = torch.empty((M, N), dtype=dt, device="cuda")
    tg.gemm(a, b[:, :320], wide, bias=None if bias is None else bias[:320], epilogue=epi)
    tg.gemm(a, b, plain, bias=bias, epilogue=epi)
    _sync_ok()
    iv = torch.int32 if c_dtype == "f32" else torch.int16
    assert torch.equal(wide.view(iv), plain[:, :320].contiguous().view(iv))
    check_dense(case, plain)


@pytest.mark.parametrize("c_dtype", [torch.bfloat16, torch.float32])
def test_wide_b_view_grouped_and_moe(c_dtype, tile):
    # the host-table grouped form (a wide 3-D view per problem) and the device-counts MoE
    # form (one 4-D view over all experts) on the same problems: bitwise equal, and parity
    counts = [0, 300, 5, 0, 130, 257, 1, 0, 64]
    case, a, b, bias, T = _moe_case(counts, 320, 200, 54, epi="bias_gelu", extra_rows=8)
    dev = torch.tensor(counts, dtype=torch.int32, device="cuda")
    out_dev = torch.full((T, 320), float("nan"), dtype=c_dtype, device="cuda")
    tg.moe_gemm_device(a, b, dev, out_dev, bias=bias, epilogue="bias_gelu")
    used = int(sum(counts))
    out_tab = torch.full((used, 320), float("nan"), dtype=c_dtype, device="cuda")
    tg.moe_grouped_gemm(a[:used], b, counts, out_tab, bias=bias, epilogue="bias_gelu")
    _sync_ok()
    iv = torch.int32 if c_dtype == torch.float32 else torch.int16
    assert torch.equal(out_dev[:used].view(iv), out_tab.view(iv))
    assert torch.isnan(out_dev[used:].float()).all(), "rows past the counts were written"
    _check_grouped(case, out_dev[:used])


# ------------------------------------------------------------------------------------------ full-size workloads

def test_workload_dense_4096_bias_gelu_full():
    case = wl.dense_case("dense_4096_bias_gelu")
    c = run_dense(case)
    _sync_ok()
    check_dense(case, c)


def test_workload_dense_8192_f32_sampled():
    case = wl.dense_case("dense_8192_f32")
    c = run_dense(case)
    _sync_ok()
    rows = sample_rows(case.M, 256, 192, seed=1)
    check_dense(case, c, rows=rows)


def test_workload_skinny_bcast_full():
    case = wl.dense_case("skinny_bcast")
    c = run_dense(case)
    _sync_ok()
    check_dense(case, c)


def test_workload_grouped_moe_sampled():
    case = wl.grouped_case("grouped_moe")
    a, b = case.a.cuda(), case.b.cuda()
    out = torch.full((a.shape[0], case.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    tg.moe_grouped_gemm(a, b, case.counts, out)
    _sync_ok()
    assert not torch.isnan(out.float()).any()
    rows = [sample_rows(int(m), 256, 24, seed=g) if m else np.zeros(0, np.int64) for g, m in enumerate(case.counts)]
    _check_grouped(case, out, rows_per_group=rows)


def test_trace_summary_of_a_small_launch():
    # the trace module's summary of a real traced launch: one unit per tile, times ordered
    from grouped_gemm_persistent_gb300 import trace
    out = trace.trace("dense_256", reps=1)
    d = out[0]
    assert d["units"] == 2 and d["pairs"] == 2                 # 2 single-CTA 128x256 tiles
    assert d["span_us"] > 0 and d["ramp_us"][0] > 0 and d["final_epi_us"][0] > 0
    assert 0.0 <= d["idle_tail_share"] < 1.0 and 0.0 < d["busy_share"] <= 1.0


# ------------------------------------------------------------------------------------------ extreme sizes

def test_long_k_integer_exact():
    # 1024 k-blocks: the operand ring laps ~170 times inside one tile; integer sums stay exact
    M, N, K = 256, 320, 65536
    case = wl.dense_random(M, N, K, seed=70, dist="int4", c_dtype="f32")
    y, _ = oracle_dense(case)
    c = run_dense(case)
    _sync_ok()
    assert np.array_equal(to_f64(c), y)


def test_tall_skinny_many_tiles_sampled():
    # 2344 M-tiles of one N-tile each: 30 rounds of the persistent schedule
    M, N, K = 600_000, 64, 64
    case = wl.dense_random(M, N, K, seed=71, dist="int4", c_dtype="f32")
    rows = np.unique(np.concatenate([sample_rows(M, 256, 64, seed=9), np.arange(M - 300, M)]))
    y, _ = oracle_dense(case, rows=rows)
    c = run_dense(case)
    _sync_ok()
    assert np.array_equal(to_f64(c[torch.as_tensor(rows, device=c.device)]), y)


def test_moe_device_counts_at_the_expert_limit():
    # TG_MOE_MAX_EXPERTS experts, a fifth of them empty, ragged counts; bitwise equal to the
    # host-table grouped GEMM and within the bound of the oracle
    G = 190
    rng = np.random.default_rng(72)
    counts = rng.integers(0, 300, size=G)
    counts[rng.choice(G, size=G // 5, replace=False)] = 0
    case, a, b, bias, T = _moe_case(counts.tolist(), 128, 64, 72)
    dev = torch.tensor(counts, dtype=torch.int32, device="cuda")
    out_dev = torch.full((T, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    tg.moe_gemm_device(a, b, dev, out_dev)
    out_tab = torch.empty_like(out_dev)
    tg.moe_grouped_gemm(a, b, counts.tolist(), out_tab)
    _sync_ok()
    assert torch.equal(out_dev.view(torch.int16), out_tab.view(torch.int16))
    _check_grouped(case, out_dev)
