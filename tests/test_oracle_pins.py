"""Pins of the CPU oracle to facts fixed outside it (no GPU needed).

Each test checks the oracle against something other than itself: values the
pages print, closed forms, brute force over every possible 2:4 mask, library
routines (numpy / torch) for the pieces that reduce to them, and invariants.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import st24_inputs as inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bits(t: torch.Tensor) -> np.ndarray:
    return inputs.raw(t.contiguous()).numpy()


# --------------------------------------------------------------- decoding pins

def test_decode_matches_torch_for_every_code():
    # Every fp16/bf16 bit pattern and every e4m3 code decodes to torch's own value.
    all16 = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    for name, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        ref = all16.view(tdt).to(torch.float64).numpy()
        got = oracle.decode(name, all16.numpy())
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), name
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode("e4m3", codes.numpy())
    assert ((got == ref) | (np.isnan(got) & np.isnan(ref))).all()
    assert got[0x7E] == 448.0 and np.isnan(got[0x7F]) and got[1] == 2.0 ** -9
    s8 = np.arange(-128, 128, dtype=np.int8)
    assert (oracle.decode("s8", s8) == s8.astype(np.float64)).all()


# ----------------------------------------------------------- worked example pin

@pytest.mark.parametrize("dt", ["f16", "bf16", "f32", "e4m3", "s8"])
def test_worked_example(dt):
    g = load("worked_example.json")
    # w0..w7 realised so that w0, w3 lead group 0 and w5, w6 lead group 1.
    w = torch.tensor([[4.0, -1.0, 0.5, -3.0, 0.25, 2.0, -5.0, 1.0]])
    W = w.to(inputs.TORCH_DTYPE[dt])
    pruned, mask, values, meta = oracle.prune_compress(dt, bits(W))
    kept = [k for k in range(g["dense_len"]) if mask[0, k]]
    assert kept == g["kept"]
    dense = oracle.decode(dt, bits(W))[0]
    pr = oracle.decode(dt, pruned)[0]
    for k in range(8):
        assert pr[k] == (dense[k] if k in g["kept"] else 0.0)
    assert list(oracle.decode(dt, values)[0]) == [dense[k] for k in g["values"]]
    idx = [[(meta[0, gi // 2] >> (4 * (gi % 2) + 2 * j)) & 3 for j in range(2)] for gi in range(2)]
    assert idx == g["indices"]
    # 2 bits per index, 4 bits per group: one metadata byte for these 2 groups.
    assert meta.shape[1] * 8 == 2 * g["bits_per_group"]


# ------------------------------------------------------- listing's printed output

def test_listing_printed_output():
    g = load("listing_output.json")
    torch.manual_seed(g["seed"])
    W = torch.randn(g["rows"], g["cols"])
    pruned, mask, values, meta = oracle.prune_compress("f32", bits(W))
    Wp = torch.from_numpy(oracle.decode("f32", pruned))
    p = g["printed"]
    assert f"{(Wp == 0).double().mean().item():.1%}" == p["sparsity"]
    groups = (Wp != 0).reshape(g["rows"], g["cols"] // 4, 4).sum(-1)
    assert str(bool((groups == 2).all().item())) == p["all groups have exactly 2 nonzeros"]
    # Byte accounting at 2 bytes per value (the page's FP16 accounting).
    M, K = g["rows"], g["cols"]
    dense_bytes = M * K * 2
    sparse_bytes = oracle.values_bytes("f16", M, K) + oracle.meta_bytes(M, K)
    assert f"{dense_bytes / 1024:.1f} KB" == p["dense"]
    assert f"{sparse_bytes / 1024:.1f} KB" == p["sparse"]
    assert f"{sparse_bytes / dense_bytes:.1%}" == p["sparse_fraction_of_dense"]
    # The compressed arrays have exactly those sizes.
    assert values.size * 2 + meta.size == sparse_bytes


def test_storage_overhead_closed_form():
    g = load("storage_overhead.json")
    M, K = 64, 1024
    for b, frac in g["metadata_fraction_of_dense"].items():
        dense_bits = M * K * int(b)
        assert oracle.meta_bytes(M, K) * 8 / dense_bits == frac
    f16 = (oracle.values_bytes("f16", M, K) + oracle.meta_bytes(M, K)) / (M * K * 2)
    assert f"{f16:.0%}" == g["fp16_compressed_fraction_of_dense_as_printed"]
    assert oracle.values_bytes("e4m3", M, K) == M * K // 2
    assert oracle.meta_row_bytes(12) == 2 and oracle.meta_row_bytes(8) == 1


# ------------------------------------------------------------ brute-force pins

def brute_force_pair(mags):
    """All 6 ways to keep 2 of 4: the largest retained magnitude, earliest pair on a tie."""
    best, best_sum = None, None
    for pair in itertools.combinations(range(4), 2):   # lexicographic order
        s = sum(mags[i] for i in pair)
        if best_sum is None or s > best_sum:
            best, best_sum = pair, s
    return best


def tie_heavy(dt, M, K, seed):
    """Inputs with many equal magnitudes, zeros and sign flips."""
    g = torch.Generator().manual_seed(seed)
    if dt == "s8":
        return torch.randint(-4, 5, (M, K), generator=g).to(torch.int8)
    vals = torch.tensor([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0, 0.25])
    pick = torch.randint(0, len(vals), (M, K), generator=g)
    return vals[pick].to(inputs.TORCH_DTYPE[dt])


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8", "f32"])
@pytest.mark.parametrize("kind", ["ties", "random"])
def test_bruteforce_all_masks(dt, kind):
    M, K = 48, 64
    if kind == "ties":
        W = tie_heavy(dt, M, K, seed=3)
    else:
        W = inputs.draw(dt, (M, K), 1.0, inputs.generator(11))
    _, mask, values, meta = oracle.prune_compress(dt, bits(W))
    mags = np.abs(oracle.decode(dt, bits(W)))
    for m in range(M):
        for gi in range(K // 4):
            pair = brute_force_pair(list(mags[m, 4 * gi:4 * gi + 4]))
            got = tuple(k for k in range(4) if mask[m, 4 * gi + k])
            assert got == pair, (m, gi, mags[m, 4 * gi:4 * gi + 4])
            nib = (meta[m, gi // 2] >> (4 * (gi % 2))) & 0xF
            assert (nib & 3, nib >> 2) == pair


def test_special_groups():
    # All-zero group keeps slots (0, 1); equal magnitudes keep the two earliest;
    # -0 ties +0; int8 -128 outranks 127; a NaN is kept.
    cases = [
        ("bf16", [0.0, 0.0, 0.0, 0.0], (0, 1)),
        ("bf16", [1.0, -1.0, 1.0, -1.0], (0, 1)),
        ("bf16", [-0.0, 0.0, 0.0, 3.0], (0, 3)),
        ("f16", [0.5, 2.0, -2.0, 2.0], (1, 2)),
        ("bf16", [1.0, float("nan"), 7.0, 2.0], (1, 2)),
        ("bf16", [float("inf"), 1.0, float("nan"), 2.0], (0, 2)),
    ]
    for dt, row, want in cases:
        W = torch.tensor([row]).to(inputs.TORCH_DTYPE[dt])
        _, mask, _, meta = oracle.prune_compress(dt, bits(W))
        assert tuple(k for k in range(4) if mask[0, k]) == want, row
        assert (meta[0, 0] & 3, (meta[0, 0] >> 2) & 3) == want
    W = torch.tensor([[-128, 127, 5, -127]], dtype=torch.int8)
    _, mask, _, _ = oracle.prune_compress("s8", W.numpy())
    assert tuple(k for k in range(4) if mask[0, k]) == (0, 1)


def test_k_not_multiple_of_4_rejected():
    with pytest.raises(ValueError):
        oracle.prune_compress("bf16", np.zeros((2, 6), np.uint16))


# ------------------------------------------------------------------ round trip

@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
@pytest.mark.parametrize("K", [4, 12, 256, 1000])
def test_decompress_of_compress_is_prune(dt, K):
    W = inputs.draw(dt, (37, K), 0.02 if dt == "e4m3" else 1.0, inputs.generator(K))
    pruned, mask, values, meta = oracle.prune_compress(dt, bits(W))
    back = oracle.decompress(dt, values, meta, K)
    assert np.array_equal(back.view(np.uint8), pruned.view(np.uint8))
    # at most 2 non-zeros per group; exactly 2 kept slots, indices ascending
    nz = (oracle.decode(dt, pruned) != 0).reshape(37, K // 4, 4).sum(-1)
    assert nz.max() <= 2
    assert (mask.reshape(37, K // 4, 4).sum(-1) == 2).all()
    nib = np.stack([meta & 0xF, meta >> 4], -1).reshape(37, -1)[:, :K // 4]
    assert ((nib & 3) < (nib >> 2)).all()


def test_exactly_two_nonzeros_on_gaussian_inputs():
    # fp16/bf16 Gaussian inputs have no zeros, so each group keeps exactly 2 non-zeros.
    for dt in ("f16", "bf16"):
        W = inputs.draw(dt, (64, 512), 0.02, inputs.generator(5))
        pruned, *_ = oracle.prune_compress(dt, bits(W))
        nz = (oracle.decode(dt, pruned) != 0).reshape(64, 128, 4).sum(-1)
        assert (nz == 2).all()


def test_decompress_rejects_invalid_metadata():
    values = np.zeros((1, 2), np.uint16)
    meta = np.array([[0x05]], np.uint8)   # indices (1, 1): not a valid pair
    with pytest.raises(ValueError):
        oracle.decompress("bf16", values, meta, 4)


# --------------------------------------------------------------------- products

@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
def test_sparse_product_equals_dense_product_of_pruned(dt):
    M, N, K = 40, 24, 96
    case = inputs.spmm_case(dt, "f32", M, N, K, a_std=0.5, seed=7)
    pruned, _, values, meta = oracle.prune_compress(dt, bits(case.A))
    Xb = bits(case.X)
    sp, sp_acc = oracle.spmm(dt, "f32", values, meta, Xb, K)
    de, de_acc = oracle.gemm_dense(dt, "f32", pruned, Xb)
    assert np.array_equal(sp, de)              # same order, exact zeros added: identical
    assert np.array_equal(sp_acc, de_acc)
    # Against a library matmul of the decoded pruned matrix.
    Ad = oracle.decode(dt, pruned)
    Bd = oracle.decode(dt, Xb)
    ref = Bd @ Ad.T                            # [N, M]
    if dt == "s8":
        iref = Xb.astype(np.int64) @ pruned.astype(np.int64).T
        assert np.array_equal(sp_acc, iref)
        assert np.array_equal(sp, iref.astype(np.float64))
    else:
        assert np.allclose(sp, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_epilogue_alpha_beta_scale():
    M, N, K = 16, 8, 32
    case = inputs.spmm_case("bf16", "bf16", M, N, K, alpha=0.75, beta=-1.5, with_scale=True, seed=2)
    _, _, values, meta = oracle.prune_compress("bf16", bits(case.A))
    acc, _ = oracle.spmm("bf16", "f32", values, meta, bits(case.X), K)
    out, _ = oracle.spmm("bf16", "bf16", values, meta, bits(case.X), K, alpha=0.75, beta=-1.5,
                         C_in=bits(case.C_in), scale=case.scale.numpy())
    cin = case.C_in.to(torch.float64).numpy()
    want = 0.75 * case.scale.numpy().astype(np.float64)[None, :] * acc - 1.5 * cin
    assert np.allclose(out, want, rtol=1e-15, atol=0)
    # beta == 0: C_in is not read (NaNs there do not matter).
    nan_c = np.full((N, M), 0x7FC0, np.uint16)
    out0, _ = oracle.spmm("bf16", "bf16", values, meta, bits(case.X), K, beta=0.0, C_in=nan_c)
    assert np.isfinite(out0).all()


def test_sampled_equals_full():
    M, N, K = 64, 16, 128
    case = inputs.spmm_case("e4m3", "bf16", M, N, K, a_std=0.02, seed=4)
    _, _, values, meta = oracle.prune_compress("e4m3", bits(case.A))
    full, _ = oracle.spmm("e4m3", "bf16", values, meta, bits(case.X), K)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, M, 50), rng.integers(0, N, 50)
    samp, _ = oracle.spmm_sampled("e4m3", "bf16", values, meta, bits(case.X), K, rows, cols)
    assert np.array_equal(samp, full[cols, rows])


def test_threads_do_not_change_results():
    M, N, K = 33, 9, 64
    case = inputs.spmm_case("f16", "f32", M, N, K, seed=9)
    _, _, values, meta = oracle.prune_compress("f16", bits(case.A))
    a, _ = oracle.spmm("f16", "f32", values, meta, bits(case.X), K, nthreads=1)
    b, _ = oracle.spmm("f16", "f32", values, meta, bits(case.X), K, nthreads=5)
    assert np.array_equal(a, b)
    assert math.isfinite(float(a.sum()))


# ---- quantise, then prune and compress (reading R7 of the oracle) ---------------

def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    """torch's own fp32 -> float8_e4m3fn cast (nearest-even), as codes."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_matches_torch():
    # every finite e4m3 value, the midpoints between neighbours (ties go to the
    # even code), the floats next to each midpoint, and a random spread over
    # the whole range including the subnormals
    vals = oracle.decode("e4m3", np.arange(256, dtype=np.uint8))
    fin = np.unique(np.abs(vals[np.isfinite(vals)])).astype(np.float64)
    mids = (fin[:-1] + fin[1:]) / 2
    rng = np.random.default_rng(5)
    xs = np.concatenate([fin, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                         np.nextafter(mids.astype(np.float32), np.float32(1000)),
                         rng.uniform(0, 448, 4000), np.exp2(rng.uniform(-12, 8.8, 4000))]).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    xs = np.concatenate([xs, -xs])
    assert np.array_equal(oracle.encode_e4m3(xs), _torch_e4m3(xs))


def test_e4m3_encoder_saturates():
    xs = np.array([448.0, 449.0, 464.0, 480.0, 1e4, 3.0e38], np.float32)
    assert list(oracle.encode_e4m3(xs)) == [0x7E] * len(xs)
    assert list(oracle.encode_e4m3(-xs)) == [0xFE] * len(xs)


def test_quantize_worked_example():
    # Row [1, -2, 3, -4, 0.5, 0.25, -0.125, 8]: amax = 8, inv = 448 / 8 = 56, so
    # the scaled row is [56, -112, 168, -224, 28, 14, -7, 448]; in e4m3 these
    # are 56 (1.75 * 2^5), -112, 160 (168 = 1.3125 * 2^7 is a tie between 1.25
    # and 1.375; the even mantissa 2 wins), -224, 28, 14, -7, 448.  Group 0
    # keeps indices 2, 3 (|160|, |224|), group 1 keeps 0, 3 (|28|, |448|).
    W = torch.tensor([[1, -2, 3, -4, 0.5, 0.25, -0.125, 8]], dtype=torch.bfloat16)
    codes, values, meta, scales = oracle.quantize_prune_compress("bf16", "e4m3", W.view(torch.uint16).numpy())
    expect = _torch_e4m3(np.array([56, -112, 160, -224, 28, 14, -7, 448], np.float32))
    assert np.array_equal(codes[0], expect)
    assert np.array_equal(values[0], expect[[2, 3, 4, 7]])
    assert meta[0, 0] == (2 | 3 << 2) | (0 | 3 << 2) << 4
    assert scales[0] == np.float32(8) / np.float32(448)
    # int8: inv = 127 / 8 = 15.875; 15.875, -31.75, 47.625, -63.5, 7.9375,
    # 3.96875, -1.984375, 127 round (ties to even) to 16, -32, 48, -64 (a tie:
    # -63.5 -> -64), 8, 4, -2, 127
    codes, values, meta, scales = oracle.quantize_prune_compress("bf16", "s8", W.view(torch.uint16).numpy())
    assert list(codes[0]) == [16, -32, 48, -64, 8, 4, -2, 127]
    assert list(values[0]) == [48, -64, 8, 127]


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("dst", ["e4m3", "s8"])
def test_quantize_against_numpy_and_torch(src, dst):
    # codes recomputed independently: numpy fp32 arithmetic for amax, inv and
    # the scaled row, torch's e4m3 cast / numpy's round-half-even for the codes;
    # then the oracle's own prune of those codes (pinned above) must give the
    # values and metadata
    g = inputs.generator(9)
    W = (torch.randn(37, 96, generator=g) * torch.exp(torch.randn(37, 1, generator=g))).to(inputs.TORCH_DTYPE[src])
    W[5] = 0
    raw = W.view(torch.uint16).numpy()
    codes, values, meta, scales = oracle.quantize_prune_compress(src, dst, raw)
    w = W.float().numpy()
    Q = np.float32(448 if dst == "e4m3" else 127)
    amax = np.abs(w).max(axis=1).astype(np.float32)
    inv = np.where(amax > 0, Q / np.where(amax > 0, amax, 1), np.float32(0)).astype(np.float32)
    y = (w * inv[:, None]).astype(np.float32)
    if dst == "e4m3":
        ref = _torch_e4m3(np.clip(y, -448, 448)).reshape(y.shape)
    else:
        ref = np.clip(np.rint(y), -127, 127).astype(np.int8)
    assert np.array_equal(codes.view(np.uint8), ref.view(np.uint8))
    assert np.array_equal(scales, np.where(amax > 0, amax / Q, 0).astype(np.float32))
    assert not codes[5].any() and scales[5] == 0
    # every non-zero row reaches the top code exactly once its absmax is scaled
    dec = oracle.decode(dst, codes).reshape(codes.shape)
    nz = amax > 0
    assert np.all(np.abs(dec[nz]).max(axis=1) == float(Q))
    _, _, v2, m2 = oracle.prune_compress(dst, codes)
    assert np.array_equal(values.view(np.uint8), v2.view(np.uint8)) and np.array_equal(meta, m2)
    # reconstruction error: half a step of the 8-bit grid, scaled back, plus
    # the fp32 roundings of inv, of the scaled value and of the scale (each a
    # relative 2^-24 of a code of at most Q: below 1e-4 of the scale)
    err = np.abs(dec * scales[:, None] - w)
    slack = 1e-4 * scales[:, None]
    if dst == "s8":
        assert np.all(err <= 0.5 * scales[:, None] + slack)
    else:
        step = np.maximum(np.abs(w) * 2.0 ** -4, 2.0 ** -10 * scales[:, None])
        assert np.all(err <= step + slack)


# ---- N:M prune written in the 2:4 form (reading R8 of the oracle) -----------------

@pytest.mark.parametrize("n,m", [(1, 4), (1, 8), (2, 8)])
@pytest.mark.parametrize("dt", ["bf16", "s8"])
def test_nm_bruteforce(dt, n, m):
    # tie-heavy rows: the kept set of every m-group maximises sum |x|, and
    # among the maximisers it is the lexicographically smallest index set
    rng = np.random.default_rng(n * 10 + m)
    vals = rng.choice([-3, -2, -1, 0, 1, 2, 3], size=(64, 8 * m))
    W = torch.tensor(vals, dtype=inputs.TORCH_DTYPE[dt])
    pruned, values, meta = oracle.prune_compress_nm(dt, n, m, inputs.raw(W).numpy())
    kept = oracle.decode(dt, pruned).reshape(pruned.shape) != 0
    mags = np.abs(vals)
    for r in range(vals.shape[0]):
        for g0 in range(0, vals.shape[1], m):
            grp = mags[r, g0:g0 + m]
            best = max(itertools.combinations(range(m), n), key=lambda c: (sum(grp[list(c)]), [-i for i in c]))
            want = np.zeros(m, bool)
            want[list(best)] = True
            # a kept zero decodes to 0: compare on the non-zero elements
            assert np.array_equal(kept[r, g0:g0 + m], want & (grp != 0))


@pytest.mark.parametrize("n,m", [(1, 4), (1, 8), (2, 8)])
@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
def test_nm_structure_and_roundtrip(dt, n, m):
    g = inputs.generator(n + m)
    W = inputs.draw(dt, (33, 16 * m), 0.02 if dt == "e4m3" else 1.0, g)
    raw = inputs.raw(W).numpy()
    pruned, values, meta = oracle.prune_compress_nm(dt, n, m, raw)
    dec = oracle.decode(dt, pruned).reshape(pruned.shape)
    # exactly n non-zeros in every m-group (no zeros in these inputs' kept slots)
    nz = (dec != 0).reshape(dec.shape[0], -1, m).sum(axis=2)
    assert np.all(nz <= n) and np.mean(nz == n) > 0.99
    # every 4-subgroup holds at most 2: the 2:4 form decompresses to the pruned matrix
    assert np.array_equal(oracle.decompress(dt, values, meta, 16 * m).view(np.uint8), pruned.view(np.uint8))
    # the pruned matrix keeps exactly the kept elements of W
    same = (pruned.view(np.uint8).reshape(dec.shape + (-1,)) == raw.view(np.uint8).reshape(dec.shape + (-1,))).all(-1)
    assert np.all(same | (dec == 0))


def test_nm_two_of_four_is_the_plain_prune():
    W = inputs.draw("bf16", (17, 64), 1.0, inputs.generator(3))
    raw = inputs.raw(W).numpy()
    p1, v1, m1 = oracle.prune_compress_nm("bf16", 2, 4, raw)
    p2, _, v2, m2 = oracle.prune_compress("bf16", raw)
    assert np.array_equal(p1, p2) and np.array_equal(v1, v2) and np.array_equal(m1, m2)


def test_nm_rejects_unsupported():
    raw = np.zeros((2, 16), np.uint16)
    for n, m in ((3, 8), (0, 4), (2, 16), (1, 3)):
        with pytest.raises(ValueError):
            oracle.prune_compress_nm("bf16", n, m, raw)


# ---- the transposed use dX = dY * W (reading R9 of the oracle) -------------------

def _small_int_case(dt, M, K, N, seed):
    """Weights and dY with small integer values (exact in every type and in fp64 sums)."""
    g = inputs.generator(seed)
    if dt == "s8":
        A = torch.randint(-9, 10, (M, K), generator=g).to(torch.int8)
        dY = torch.randint(-9, 10, (N, M), generator=g).to(torch.int8)
    else:
        A = torch.randint(-9, 10, (M, K), generator=g).to(torch.float32).to(inputs.TORCH_DTYPE[dt])
        dY = torch.randint(-9, 10, (N, M), generator=g).to(torch.float32).to(inputs.TORCH_DTYPE[dt])
    return bits(A), bits(dY)


@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
def test_transposed_adjoint_of_the_forward_product(dt):
    """<y, A x> == <A^T y, x> exactly: the transposed product is the adjoint of the
    forward one (an index slip, a swapped i0/i1 or a transposed operand breaks it)."""
    M, K = 48, 64
    A, _ = _small_int_case(dt, M, K, 1, 3)
    _, _, values, meta = oracle.prune_compress(dt, A)
    g = inputs.generator(11)
    for _ in range(3):
        if dt == "s8":
            x = torch.randint(-5, 6, (1, K), generator=g).to(torch.int8)
            y = torch.randint(-5, 6, (1, M), generator=g).to(torch.int8)
        else:
            x = torch.randint(-5, 6, (1, K), generator=g).to(torch.float32).to(inputs.TORCH_DTYPE[dt])
            y = torch.randint(-5, 6, (1, M), generator=g).to(torch.float32).to(inputs.TORCH_DTYPE[dt])
        Ax, _ = oracle.spmm(dt, "f32", values, meta, bits(x), K)          # [1, M]
        Aty, _ = oracle.spmm_t(dt, "f32", values, meta, bits(y), K)       # [1, K]
        lhs = float(oracle.decode(dt, bits(y))[0] @ Ax[0])
        rhs = float(Aty[0] @ oracle.decode(dt, bits(x))[0])
        assert lhs == rhs


@pytest.mark.parametrize("dt", ["f16", "bf16", "s8"])
def test_transposed_equals_matmul_of_the_decompressed_weight(dt):
    M, K, N = 40, 96, 12
    case = inputs.spmm_case(dt, "f32", M, N, K, a_std=0.5, seed=8)
    g = inputs.generator(21)
    dY = inputs.draw(dt, (N, M), 1.0, g)
    _, _, values, meta = oracle.prune_compress(dt, bits(case.A))
    out, acc = oracle.spmm_t(dt, "f32", values, meta, bits(dY), K)
    dense = oracle.decompress(dt, values, meta, K)                       # [M, K]
    if dt == "s8":
        ref = bits(dY).astype(np.int64) @ dense.astype(np.int64)          # [N, K]
        assert np.array_equal(acc, ref)
        assert np.array_equal(out, ref.astype(np.float64))
    else:
        ref = oracle.decode(dt, bits(dY)) @ oracle.decode(dt, dense)
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_transposed_epilogue_and_sampling():
    M, K, N = 32, 64, 8
    A, dY = _small_int_case("bf16", M, K, N, 5)
    _, _, values, meta = oracle.prune_compress("bf16", A)
    acc, _ = oracle.spmm_t("bf16", "f32", values, meta, dY, K)
    g = inputs.generator(6)
    cin = inputs.draw("bf16", (N, K), 1.0, g)
    out, _ = oracle.spmm_t("bf16", "bf16", values, meta, dY, K, alpha=0.5, beta=-2.0, C_in=bits(cin))
    assert np.array_equal(out, 0.5 * acc - 2.0 * cin.to(torch.float64).numpy())
    rng = np.random.default_rng(1)
    ks, ns = rng.integers(0, K, 40), rng.integers(0, N, 40)
    samp, _ = oracle.spmm_t_sampled("bf16", "bf16", values, meta, dY, K, ks, ns, alpha=0.5, beta=-2.0,
                                    C_in=bits(cin))
    assert np.array_equal(samp, out[ns, ks])


# ---- N:M with up to four kept per subgroup, as two 2:4 forms (reading R10) --------

@pytest.mark.parametrize("n", [3, 4])
@pytest.mark.parametrize("dt", ["bf16", "s8"])
def test_nm2_bruteforce(dt, n):
    # tie-heavy rows: the kept set of every 8-group maximises sum |x|, the
    # lexicographically smallest index set among the maximisers
    m = 8
    rng = np.random.default_rng(n)
    vals = rng.choice([-3, -2, -1, 0, 1, 2, 3], size=(64, 64))
    W = torch.tensor(vals, dtype=inputs.TORCH_DTYPE[dt])
    pruned, values, meta = oracle.prune_compress_nm2(dt, n, m, inputs.raw(W).numpy())
    kept = oracle.decode(dt, pruned).reshape(pruned.shape) != 0
    mags = np.abs(vals)
    for r in range(vals.shape[0]):
        for g0 in range(0, vals.shape[1], m):
            grp = mags[r, g0:g0 + m]
            best = max(itertools.combinations(range(m), n), key=lambda c: (sum(grp[list(c)]), [-i for i in c]))
            want = np.zeros(m, bool)
            want[list(best)] = True
            assert np.array_equal(kept[r, g0:g0 + m], want & (grp != 0))


@pytest.mark.parametrize("n,m", [(4, 8), (3, 8), (2, 8), (1, 4), (4, 4)])
@pytest.mark.parametrize("dt", ["f16", "bf16", "e4m3", "s8"])
def test_nm2_two_forms_sum_to_the_pruned_matrix(dt, n, m):
    K = 16 * m
    W = inputs.draw(dt, (29, K), 1.0, inputs.generator(n * m))
    raw = inputs.raw(W).numpy()
    pruned, values, meta = oracle.prune_compress_nm2(dt, n, m, raw)
    mrb = oracle.meta_row_bytes(K)
    # each half is a valid 2:4 form (ascending index pairs), and the two add up to the pruned matrix
    f0 = oracle.decompress(dt, np.ascontiguousarray(values[:, :K // 2]), np.ascontiguousarray(meta[:, :mrb]), K)
    f1 = oracle.decompress(dt, np.ascontiguousarray(values[:, K // 2:]), np.ascontiguousarray(meta[:, mrb:]), K)
    total = oracle.decode(dt, f0) + oracle.decode(dt, f1)
    assert np.array_equal(total, oracle.decode(dt, pruned))
    # no position holds a non-zero in both forms
    assert not np.any((oracle.decode(dt, f0) != 0) & (oracle.decode(dt, f1) != 0))
    # exactly n non-zeros per m-group on inputs without zeros among the kept
    nz = (oracle.decode(dt, pruned) != 0).reshape(29, -1, m).sum(axis=2)
    assert np.all(nz <= n) and np.mean(nz == n) > 0.95
    # with n <= 2, form 0 is the one-form result and form 1 is all zeros
    if n <= 2 and m in (4, 8):
        p1, v1, m1 = oracle.prune_compress_nm(dt, n, m, raw)
        assert np.array_equal(values[:, :K // 2].view(np.uint8), v1.view(np.uint8))
        assert np.array_equal(meta[:, :mrb], m1)
        assert not np.any(oracle.decode(dt, f1))


def test_nm2_product_over_the_stacked_forms():
    """The two forms as one M x 2K 2:4 matrix times B stacked twice equal the pruned
    matrix times B (integer-valued inputs: every sum exact in fp64)."""
    K, M, N = 64, 24, 5
    g = inputs.generator(8)
    A = torch.randint(-9, 10, (M, K), generator=g).to(torch.float32).to(torch.bfloat16)
    X = torch.randint(-9, 10, (N, K), generator=g).to(torch.float32).to(torch.bfloat16)
    pruned, values, meta = oracle.prune_compress_nm2("bf16", 4, 8, bits(A))
    X2 = np.concatenate([bits(X), bits(X)], axis=1)          # [N, 2K]: B stacked twice along K
    sp, _ = oracle.spmm("bf16", "f32", values, meta, X2, 2 * K)
    de, _ = oracle.gemm_dense("bf16", "f32", pruned, bits(X))
    assert np.array_equal(sp, de)


def test_nm2_rejects_unsupported():
    W = np.zeros((4, 64), np.uint16)
    for n, m in [(5, 8), (0, 8), (2, 16), (3, 2)]:
        with pytest.raises(ValueError):
            oracle.prune_compress_nm2("bf16", n, m, W)
