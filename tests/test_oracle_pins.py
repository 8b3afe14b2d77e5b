"""Pins for the float64 oracle, checked against things other than itself.

Each test ties the oracle to something it does not contain: a library dtype
cast, the OCP element tables, a worked property from the pages, a closed form
worked by hand, an invariant of the mathematics, or the same computation taken
through numpy's einsum on independently decoded values. They are chosen so a
dropped term, a wrong sign, a wrong index or a transposed operand in
oracle/dsa_oracle.c fails at least one of them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from infra_dsa_indexer_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

FMTS = [synth.FMT_BF16, synth.FMT_E4M3, synth.FMT_MXFP8, synth.FMT_MXFP4]


def run(case, **kw):
    return oracle.logits(case.fmt, case.q, case.k, case.w, case.ks, case.ke,
                         case.sm_scale, q_sf=case.q_sf, k_sf=case.k_sf,
                         k_tok=case.k_tok, w_fmt=case.w_fmt, H=case.H, D=case.D,
                         **kw)


# ---------------------------------------------------------------------------
# decoders vs library casts and the OCP tables
# ---------------------------------------------------------------------------

def _same(a, b):
    return (np.isnan(a) and np.isnan(b)) or a == b


def test_decode_bf16_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for c in range(0, 65536, 1):
        got = oracle.decode_bf16(int(c))
        assert _same(got, ref[c]), (hex(c), got, ref[c])


def test_decode_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        assert _same(oracle.decode_e4m3(c), ref[c]), hex(c)
    assert oracle.decode_e4m3(0x7E) == 448.0          # OCP max normal
    assert oracle.decode_e4m3(0x01) == 2.0 ** -9       # smallest subnormal


def test_decode_e8m0_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(256):
        assert _same(oracle.decode_e8m0(c), ref[c]), hex(c)
    assert oracle.decode_e8m0(0x7F) == 1.0            # "MX scales are one"


def test_decode_e2m1_matches_ocp_table():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_table.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, val = line.split()
                table[int(code, 2)] = float(val)
    assert len(table) == 16
    for c, v in table.items():
        assert oracle.decode_e2m1(c) == v, (bin(c), v)


# ---------------------------------------------------------------------------
# independent decoders for the library route
# ---------------------------------------------------------------------------

_E2M1_MAG = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def _dequant_lib(fmt, x, sf, D):
    """Dequantise with torch casts (bf16, e4m3, e8m0) and the OCP E2M1 table."""
    if fmt == synth.FMT_BF16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    if fmt == synth.FMT_MXFP4:
        lo = x & 0xF
        hi = x >> 4
        codes = np.stack([lo, hi], axis=-1).reshape(*x.shape[:-1], D)
        vals = _E2M1_MAG[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    else:
        vals = torch.from_numpy(x).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if fmt in (synth.FMT_MXFP8, synth.FMT_MXFP4):
        s = torch.from_numpy(sf).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        vals = vals * np.repeat(s, 32, axis=-1)
    return vals


def library_route(case):
    qd = _dequant_lib(case.fmt, case.q, case.q_sf, case.D)           # [B,S,H,D]
    kd = _dequant_lib(case.fmt, case.k, case.k_sf, case.D)           # [B,N,D]
    if case.k_tok is not None:
        kd = kd * case.k_tok.astype(np.float64)[..., None]
    if case.w_fmt == synth.W_BF16:
        w = _dequant_lib(synth.FMT_BF16, case.w, None, None)
    else:
        w = case.w.astype(np.float64)
    dots = np.einsum("bshd,bnd->bshn", qd, kd)                        # [B,S,H,N]
    x = case.sm_scale * dots
    out = np.einsum("bsh,bshn->bsn", w, np.maximum(x, 0.0))
    den = np.einsum("bsh,bshn->bsn", np.abs(w), np.abs(x))
    # the looser scale: sum_h |w_h| |sm_scale| sum_d |q_hd| |k_d|
    den_abs = abs(case.sm_scale) * np.einsum(
        "bsh,bshn->bsn", np.abs(w), np.einsum("bshd,bnd->bshn", np.abs(qd), np.abs(kd)))
    cols = np.arange(case.N)
    lo = np.clip(case.ks, 0, case.N)[..., None]
    hi = np.clip(case.ke, 0, case.N)[..., None]
    inside = (cols >= lo) & (cols < hi)
    out = np.where(inside, out, -np.inf)
    return (out.reshape(-1, case.N), np.where(inside, den, 0).reshape(-1, case.N),
            np.where(inside, den_abs, 0).reshape(-1, case.N))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("w_fmt", [synth.W_F32, synth.W_BF16])
def test_library_route_agrees(fmt, w_fmt):
    """numpy einsum over torch-decoded values == the C loops, to float64 rounding."""
    rng = np.random.default_rng(fmt * 7 + w_fmt)
    B, S, N, H = 2, 4, 40, 3
    ks = rng.integers(-3, N // 2, size=(B, S))
    ke = ks + rng.integers(-2, N, size=(B, S))
    case = synth.make_case(fmt, B, S, N, H=H, D=128, seed=11 + fmt, ks=ks, ke=ke,
                           w_fmt=w_fmt, sm_scale=0.37)
    out, den, den_abs = run(case, want_den_abs=True)
    ref, rden, rden_abs = library_route(case)
    assert np.array_equal(np.isneginf(out), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.all(np.abs(out[fin] - ref[fin]) <= 1e-12 * (1e-300 + rden[fin]) + 1e-300)
    assert np.allclose(den[fin], rden[fin], rtol=1e-12, atol=0)
    assert np.allclose(den_abs[fin], rden_abs[fin], rtol=1e-12, atol=0)
    assert np.all(den_abs[~fin] == 0) and np.all(den[~fin] == 0)
    # |sum_d q k| <= sum_d |q||k| head by head, so den <= den_abs
    assert np.all(den[fin] <= den_abs[fin] * (1 + 1e-12))


# ---------------------------------------------------------------------------
# the pages' own worked property: all-zero inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_zero_inputs_reproducer_property(fmt):
    """The DeepGEMM reproducer's check: all-zero Q/K/W with MX scales of one,
    windows [0, n-m+row); -inf exactly where not (col < end), 0 elsewhere."""
    m, n = 12, 40
    case = synth.make_case(fmt, 1, m, n, H=4, seed=0, zero=True, windows="causal_excl")
    out, _, _ = run(case)
    cols = np.arange(n)[None, :]
    ends = (np.arange(m) + n - m)[:, None]
    valid = cols < ends
    assert np.array_equal(np.isneginf(out), ~valid)
    assert np.all(out[valid] == 0.0)


def test_zero_mask_golden_fixture():
    """Stored mask for m=4, n=8 written from the reproducer's window rule."""
    with open(os.path.join(GOLDEN, "zero_inputs_mask_m4_n8.txt")) as f:
        rows = [l.split("#")[0].strip() for l in f]
    rows = [r for r in rows if r]
    mask = np.array([[c == "x" for c in r] for r in rows])
    case = synth.make_case(synth.FMT_MXFP8, 1, 4, 8, H=2, zero=True, windows="causal_excl")
    out, _, _ = run(case)
    assert np.array_equal(np.isneginf(out), mask)


# ---------------------------------------------------------------------------
# closed forms worked by hand
# ---------------------------------------------------------------------------

def _bf16_case_from_values(qv, kv, wv, sm_scale, ks, ke):
    B, S, H, D = qv.shape
    N = kv.shape[1]
    case = synth.make_case(synth.FMT_BF16, B, S, N, H=H, D=D, ks=ks, ke=ke,
                           sm_scale=sm_scale)
    case.q = synth.to_bf16_codes(qv)
    case.k = synth.to_bf16_codes(kv)
    case.w = wv.astype(np.float32)
    return case


def test_one_hot_closed_form():
    """q[i,h,:] = c_h e_{d_h}, k[j,:] = a_j e_{d_j}: the dot is c_h a_j when
    d_h == d_j else 0, so logits = sum_h w_h max(0, s c_h a_j [d_h == d_j])."""
    H, D, N = 3, 128, 5
    c = np.array([2.0, -1.5, 0.5])
    dh = np.array([7, 7, 100])
    a = np.array([1.0, -2.0, 4.0, 0.5, 3.0])
    dj = np.array([7, 7, 100, 3, 100])
    w = np.array([0.25, -1.0, 2.0])
    s = 0.5
    qv = np.zeros((1, 1, H, D), np.float32)
    for h in range(H):
        qv[0, 0, h, dh[h]] = c[h]
    kv = np.zeros((1, N, D), np.float32)
    for j in range(N):
        kv[0, j, dj[j]] = a[j]
    wv = w.reshape(1, 1, H)
    case = _bf16_case_from_values(qv, kv, wv, s, [[0]], [[N]])
    out, _, _ = run(case)
    # by hand:
    # j=0 (a=1, d=7):   h0: .25*max(0,.5*2*1)=.25 ; h1: -1*max(0,.5*-1.5)=0 ; h2: d mismatch -> 0
    # j=1 (a=-2, d=7):  h0: max(0,-2)=0 ; h1: -1*max(0,.5*-1.5*-2=1.5)=-1.5
    # j=2 (a=4, d=100): h2: 2*max(0,.5*.5*4=1)=2
    # j=3 (d=3): 0
    # j=4 (a=3, d=100): h2: 2*max(0,.5*.5*3=.75)=1.5
    assert out[0].tolist() == [0.25, -1.5, 2.0, 0.0, 1.5]


def test_single_head_textbook_dot():
    """H=1, w=1, s>0 reduces to ReLU(s * q.k), a plain dot product."""
    rng = np.random.default_rng(5)
    qv = rng.standard_normal((1, 3, 1, 128)).astype(np.float32)
    kv = rng.standard_normal((1, 7, 128)).astype(np.float32)
    case = _bf16_case_from_values(qv, kv, np.ones((1, 3, 1)), 0.125, [[0] * 3], [[7] * 3])
    out, _, _ = run(case)
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy()[0, :, 0]
    kd = torch.from_numpy(case.k.view(np.int16)).view(torch.bfloat16).double().numpy()[0]
    ref = np.maximum(0.125 * (qd @ kd.T), 0.0)
    assert np.allclose(out, ref, rtol=1e-14, atol=0)


def test_fp4_nibble_order():
    """Element 2k sits in the low nibble: a one-hot 1.0 (code 0b0010) at d=2
    is byte 1 = 0x02, at d=3 it is 0x20."""
    H, D, N = 1, 32, 2
    for d in (2, 3):
        case = synth.make_case(synth.FMT_MXFP4, 1, 1, N, H=H, D=D, ks=[[0]], ke=[[N]],
                               sm_scale=1.0, mx_unit_scales=True, zero=True)
        case.q = np.zeros((1, 1, 1, D // 2), np.uint8)
        case.q[0, 0, 0, d // 2] = 0x02 if d % 2 == 0 else 0x20
        case.k = np.zeros((1, N, D // 2), np.uint8)
        case.k[0, 0, 1] = 0x02     # k0 = e_2
        case.k[0, 1, 1] = 0x20     # k1 = e_3
        case.w = np.ones((1, 1, 1), np.float32)
        out, _, _ = run(case)
        expect = [1.0, 0.0] if d == 2 else [0.0, 1.0]
        assert out[0].tolist() == expect


def test_fp4_row_dequant_nibble_order_and_blocks():
    """Byte b of an E2M1 row holds element 2b in its low nibble and 2b+1 in
    its high nibble (the torch float4_e2m1fn_x2 packing); element d takes the
    E8M0 scale of block d // 32."""
    D = 64
    data = np.zeros(D // 2, np.uint8)
    data[0] = 0x3A        # d0 = code 0xA (-1.0), d1 = code 0x3 (1.5)
    data[20] = 0x71       # d40 = code 0x1 (0.5), d41 = code 0x7 (6.0)
    sf = np.array([0x7F + 1, 0x7F - 2], np.uint8)     # x2, x0.25
    got = oracle.dequant_row(synth.FMT_MXFP4, data, sf, D)
    expect = np.zeros(D)
    expect[0], expect[1] = -1.0 * 2, 1.5 * 2
    expect[40], expect[41] = 0.5 * 0.25, 6.0 * 0.25
    assert np.array_equal(got, expect)


def test_mx_block_scale_locality():
    """The E8M0 byte of block b scales only dims 32b..32b+31."""
    D, N = 128, 4
    case = synth.make_case(synth.FMT_MXFP8, 1, 1, N, H=1, D=D, ks=[[0]], ke=[[N]],
                           sm_scale=1.0, zero=True, mx_unit_scales=True)
    q = np.zeros((1, 1, 1, D), np.uint8)
    q[0, 0, 0, :] = 0x38                   # e4m3 1.0 everywhere
    k = np.zeros((1, N, D), np.uint8)
    for j in range(N):
        k[0, j, 32 * j + 5] = 0x38         # key j: 1.0 at one dim of block j
    case.q, case.k = q, k
    case.w = np.ones((1, 1, 1), np.float32)
    case.k_sf = np.full((1, N, 4), 0x7F, np.uint8)
    case.k_sf[0, :, 2] = 0x7F + 3          # block 2 of every key: x8
    case.q_sf = np.full((1, 1, 1, 4), 0x7F, np.uint8)
    case.q_sf[0, 0, 0, 1] = 0x7F - 1       # block 1 of the query: x0.5
    out, _, _ = run(case)
    assert out[0].tolist() == [1.0, 0.5, 8.0, 1.0]


def test_fp8_per_token_scale_multiplies_key():
    D, N = 128, 3
    case = synth.make_case(synth.FMT_E4M3, 1, 1, N, H=1, D=D, ks=[[0]], ke=[[N]],
                           sm_scale=1.0, seed=1)
    case.q = np.zeros((1, 1, 1, D), np.uint8)
    case.q[0, 0, 0, 9] = 0x40                  # e4m3 2.0
    case.k = np.zeros((1, N, D), np.uint8)
    case.k[0, :, 9] = 0x38                     # 1.0
    case.k_tok = np.array([[0.5, 3.0, 0.0]], np.float32)
    case.w = np.array([[[1.5]]], np.float32)
    out, _, _ = run(case)
    assert out[0].tolist() == [1.5 * 2.0 * 0.5, 1.5 * 2.0 * 3.0, 0.0]


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_zero_w_gives_zero(fmt):
    case = synth.make_case(fmt, 1, 4, 33, H=8, seed=3)
    case.w = np.zeros_like(case.w)
    out, _, _ = run(case)
    assert np.all(out == 0.0)


@pytest.mark.parametrize("fmt", FMTS)
def test_nonnegative_w_gives_nonnegative_logits(fmt):
    case = synth.make_case(fmt, 1, 4, 50, H=8, seed=4, windows="causal")
    case.w = np.abs(case.w)
    out, den, _ = run(case)
    fin = np.isfinite(out)
    assert np.all(out[fin] >= 0.0)
    assert np.all(out[fin] <= den[fin] * (1 + 1e-15))


@pytest.mark.parametrize("fmt", FMTS)
def test_linearity_in_w(fmt):
    """f(a W1 + b W2) = a f(W1) + b f(W2). The weights are multiples of 1/64
    below 2 in magnitude, so a*W1 + b*W2 is exact in float32."""
    case = synth.make_case(fmt, 1, 4, 45, H=8, seed=5)
    rng = np.random.default_rng(9)
    w1 = (rng.integers(-128, 128, case.w.shape) / 64.0).astype(np.float32)
    w2 = (rng.integers(-128, 128, case.w.shape) / 64.0).astype(np.float32)
    a, b = 0.75, -2.5
    case.w = w1
    o1, d1, _ = run(case)
    case.w = w2
    o2, d2, _ = run(case)
    case.w = (np.float32(a) * w1 + np.float32(b) * w2).astype(np.float32)
    assert np.array_equal(case.w.astype(np.float64),
                          a * w1.astype(np.float64) + b * w2.astype(np.float64))
    o3, d3, _ = run(case)
    fin = np.isfinite(o3)
    tol = 1e-12 * (abs(a) * d1 + abs(b) * d2 + d3)[fin] + 1e-300
    assert np.all(np.abs(o3[fin] - (a * o1 + b * o2)[fin]) <= tol)


@pytest.mark.parametrize("fmt", FMTS)
def test_head_permutation_invariance(fmt):
    case = synth.make_case(fmt, 1, 3, 30, H=6, seed=6)
    out, den, _ = run(case)
    perm = np.array([3, 0, 5, 1, 4, 2])
    case.q = case.q[:, :, perm]
    case.w = case.w[:, :, perm]
    if case.q_sf is not None:
        case.q_sf = case.q_sf[:, :, perm]
    out2, _, _ = run(case)
    fin = np.isfinite(out)
    assert np.array_equal(np.isneginf(out), np.isneginf(out2))
    assert np.all(np.abs(out[fin] - out2[fin]) <= 1e-13 * den[fin] + 1e-300)


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP8, synth.FMT_MXFP4])
def test_mx_scale_positive_homogeneity(fmt):
    """Raising every K E8M0 byte by e multiplies the logits by exactly 2^e."""
    case = synth.make_case(fmt, 1, 4, 40, H=4, seed=7)
    case.k_sf = np.clip(case.k_sf, 0, 240).astype(np.uint8)
    out, _, _ = run(case)
    case.k_sf = (case.k_sf + 3).astype(np.uint8)
    out2, _, _ = run(case)
    fin = np.isfinite(out)
    assert np.array_equal(out2[fin], out[fin] * 8.0)


def test_sm_scale_homogeneity_and_sign():
    case = synth.make_case(synth.FMT_BF16, 1, 4, 40, H=4, seed=8, sm_scale=0.25)
    out, _, _ = run(case)
    case.sm_scale = 0.5
    out2, _, _ = run(case)
    fin = np.isfinite(out)
    assert np.array_equal(out2[fin], 2.0 * out[fin])
    # s < 0: ReLU(s*q.k) = ReLU(|s| * q.(-k)); negating bf16 is a sign-bit flip
    case.sm_scale = -0.25
    out3, _, _ = run(case)
    case.sm_scale = 0.25
    case.k = (case.k ^ np.uint16(0x8000)).astype(np.uint16)
    out4, _, _ = run(case)
    assert np.array_equal(out3[fin], out4[fin])


def test_mx_unit_scales_equal_plain_e4m3():
    case = synth.make_case(synth.FMT_MXFP8, 1, 4, 40, H=4, seed=9, mx_unit_scales=True)
    out, _, _ = run(case)
    plain = synth.make_case(synth.FMT_E4M3, 1, 4, 40, H=4, seed=9)
    plain.q, plain.k, plain.w, plain.k_tok = case.q, case.k, case.w, None
    out2, _, _ = run(plain)
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP8, synth.FMT_MXFP4])
def test_mx_equals_bf16_of_dequantised(fmt):
    """Dequantised MX values are exactly bf16: same inputs, same float64 result."""
    case = synth.make_case(fmt, 1, 4, 36, H=4, seed=10)
    out, _, _ = run(case)
    qd = _dequant_lib(fmt, case.q, case.q_sf, case.D).astype(np.float32)
    kd = _dequant_lib(fmt, case.k, case.k_sf, case.D).astype(np.float32)
    b = synth.make_case(synth.FMT_BF16, 1, 4, 36, H=4, seed=10)
    b.q, b.k, b.w = synth.to_bf16_codes(qd), synth.to_bf16_codes(kd), case.w
    assert np.array_equal(_dequant_lib(synth.FMT_BF16, b.q, None, None), qd.astype(np.float64))
    out2, _, _ = run(b)
    assert np.array_equal(out, out2)


# ---------------------------------------------------------------------------
# the mask
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 127, 129, 999])
def test_mask_ragged_and_degenerate_windows(N):
    S = 8
    ks = np.array([[0, -5, 3, 7, N, N - 1, 4, 0]])
    ke = np.array([[N, N + 9, 3, 2, N + 3, N, 4 + N // 2, 1]])
    case = synth.make_case(synth.FMT_BF16, 1, S, N, H=2, seed=N, ks=ks, ke=ke)
    out, _, _ = run(case)
    cols = np.arange(N)
    for i in range(S):
        lo, hi = max(ks[0, i], 0), min(ke[0, i], N)
        expect = (cols < lo) | (cols >= hi)
        assert np.array_equal(np.isneginf(out[i]), expect), i
        assert np.all(np.isfinite(out[i][~expect]))


def test_row_subset_matches_full():
    case = synth.make_case(synth.FMT_E4M3, 2, 8, 64, H=4, seed=12, windows="causal")
    full, den, _ = run(case)
    rows = np.array([15, 0, 9, 3], dtype=np.int64)
    sub, dsub, _ = run(case, rows=rows)
    assert np.array_equal(sub, full[rows])
    assert np.array_equal(dsub, den[rows])
