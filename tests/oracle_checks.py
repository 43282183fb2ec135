"""Pins of the fp64 oracle against things other than itself.

Each ``check_*`` function raises AssertionError on failure.  They are run by
``test_oracle_pins.py`` against the in-tree oracle, and by
``test_oracle_mutants.py`` against deliberately broken copies of the oracle
source, each of which must fail at least one check.

What the checks compare the oracle with:
  * library routines in fp64: torch.nn.functional.rms_norm,
    torch.nn.functional.scaled_dot_product_attention, torch's float8_e4m3fn
    cast, numpy complex exponentials (RoPE written as a complex rotation);
  * closed forms and special cases: constant inputs to RMSNorm, RoPE at
    position zero, a hand-worked single-pair rotation per axis, constant V,
    zero Q (uniform attention), a single token, a ones column in V (softmax
    rows sum to one), a hand-worked two-token head;
  * invariants: per-pair norms under RoPE, the output under a common shift
    of every position on one axis, permutation equivariance over tokens;
  * the E4M3 code table: every one of the 254 finite codes round-trips,
    midpoints round to the even code, out-of-range values saturate;
  * the QKV projection: numpy's fp64 matmul (with torch rms_norm and the
    complex-rotation RoPE on its Q and K parts), identity weights (the
    prologue of x itself), a zero weight matrix (the bias alone);
  * the VC-Attention repair (reading R7): a brute-force restatement from the
    library routines (torch rms_norm, complex RoPE, torch's E4M3 cast, a
    Python sort of (error, index) pairs, torch SDPA); rho = 0 is plain FP8
    attention bit for bit, rho = 1 is SDPA over the dequantised Q' and the
    exact K', V; equal errors go to the lower token index; a planted
    badly-quantised token is always selected;
  * the Sol-Attention block mask (reading R8): pooled means, block masses
    and the keep rule restated with torch's softmax; tau = 0 is dense
    attention; a tau that keeps one block per query block is torch SDPA over
    that block's keys alone.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from synthetic import bf16_bits_from_f32, bf16_bits_to_f32, position_ids

AX = (16, 56, 56)
THETA = 10000.0
EPS = 1e-6
D = 128


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------- library references

def lib_rms(x: np.ndarray, w: np.ndarray, eps: float = EPS) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float64))
    return F.rms_norm(t, (x.shape[-1],), weight=torch.from_numpy(np.asarray(w, np.float64)),
                      eps=eps).numpy()


def lib_rope(y: np.ndarray, pos: np.ndarray, theta: float = THETA, axes=AX) -> np.ndarray:
    """RoPE as complex rotation: pair (y_2j, y_2j+1) of axis block a is the complex
    number y_2j + i y_2j+1 multiplied by exp(i pos_a theta^(-2j/d_a))."""
    B, N, H, d = y.shape
    ang = []
    for a, da in enumerate(axes):
        j = np.arange(da // 2, dtype=np.float64)
        freq = np.exp(-np.log(theta) * 2.0 * j / da)
        ang.append(pos[:, a:a + 1].astype(np.float64) * freq[None, :])
    ang = np.concatenate(ang, 1)                              # [N, d/2]
    z = y[..., 0::2] + 1j * y[..., 1::2]
    z = z * np.exp(1j * ang)[None, :, None, :]
    out = np.empty_like(y)
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def lib_attention(qn: np.ndarray, kn: np.ndarray, v: np.ndarray) -> np.ndarray:
    """torch SDPA (fp64, CPU) on [B, N, H, d] arrays, returns [B, N, H, d]."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float64)).permute(0, 2, 1, 3)
    o = F.scaled_dot_product_attention(t(qn), t(kn), t(v))
    return o.permute(0, 2, 1, 3).contiguous().numpy()


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert err <= tol, "%s: max abs err %.3e > %.1e" % (what, err, tol)


# ------------------------------------------------------------------ E4M3

def check_e4m3_exhaustive_roundtrip():
    codes = np.arange(256, dtype=np.uint8)
    finite = codes[(codes & 0x7F) != 0x7F]
    assert finite.size == 254
    dec = oracle.e4m3_decode(finite)
    assert np.all(np.isfinite(dec))
    enc = oracle.e4m3_encode(dec)
    assert np.array_equal(enc, finite), "E4M3 code does not round-trip"
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    # the decoded table is the torch float8_e4m3fn table
    tv = torch.from_numpy(finite.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(dec, tv), "E4M3 decode differs from torch's table"


def check_e4m3_matches_torch_cast():
    rng = _rng(3)
    mag = np.exp2(rng.uniform(-12.0, math.log2(463.0), 20000))
    x = mag * rng.choice([-1.0, 1.0], mag.size)
    ours = oracle.e4m3_decode(oracle.e4m3_encode(x))
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs), "E4M3 rounding differs from torch's cast"


def check_e4m3_ties_and_saturation():
    cases = {
        1.0625: 1.0,            # midpoint of 1.0 (m=0) and 1.125 (m=1) -> even m=0
        1.1875: 1.25,           # midpoint of m=1 and m=2 -> m=2
        2.0 ** -10: 0.0,        # half the smallest subnormal -> 0
        3 * 2.0 ** -10: 2 * 2.0 ** -9,   # midpoint of 1 and 2 subnormal units -> 2
        15 * 2.0 ** -10: 2.0 ** -6,      # midpoint of 7 units and the smallest normal -> normal
        440.0: 448.0,           # midpoint of 416 and 448 -> m=6 (even)
        447.9: 448.0,
        463.99: 448.0,          # saturate
        1e6: 448.0,
        -1e6: -448.0,
        0.0: 0.0,
    }
    for x, want in cases.items():
        got = float(oracle.e4m3_decode(oracle.e4m3_encode(np.array([x])))[0])
        assert got == want, "E4M3(%r) = %r, want %r" % (x, got, want)


# --------------------------------------------------------------- RMSNorm

def check_rmsnorm_matches_torch():
    rng = _rng(4)
    x = rng.standard_normal((2, 9, 3, D)) * rng.uniform(0.01, 30.0, (2, 9, 3, 1))
    w = 1.0 + 0.1 * rng.standard_normal(D)
    pos = np.zeros((9, 3), np.int32)          # RoPE is the identity at position 0
    got = oracle.prologue(x, pos, w)
    _close(got, lib_rms(x, w), 1e-12, "RMSNorm vs torch rms_norm")


def check_rmsnorm_closed_form():
    for c in (1.0, -3.0, 1e-4, 0.0):
        x = np.full((1, 1, 1, D), c)
        w = np.linspace(0.5, 1.5, D)
        got = oracle.prologue(x, np.zeros((1, 3), np.int32), w)[0, 0, 0]
        want = c / math.sqrt(c * c + EPS) * w
        _close(got, want, 1e-13, "RMSNorm of a constant row (c=%g)" % c)


# ------------------------------------------------------------------ RoPE

def check_rope_complex_form():
    rng = _rng(5)
    N = 11
    x = rng.standard_normal((1, N, 2, D))
    w = 1.0 + 0.1 * rng.standard_normal(D)
    pos = rng.integers(-50, 200, (N, 3)).astype(np.int32)
    got = oracle.prologue(x, pos, w)
    want = lib_rope(lib_rms(x, w), pos)
    _close(got, want, 1e-11, "RoPE vs complex rotation")


def check_rope_hand_cases():
    """Single nonzero element e_i, w = 1: after RMSNorm it is u = 1/sqrt(1/d + eps);
    the pair containing it turns by the hand-computed angle."""
    u = 1.0 / math.sqrt(1.0 / D + EPS)
    cases = [
        # (dim, pos, angle)
        (0, (1, 0, 0), 1.0),                                   # axis 0, pair 0, freq 1
        (2, (5, 0, 0), 5.0 * THETA ** (-2.0 / 16)),            # axis 0, pair 1
        (16, (0, 1, 0), 1.0),                                  # axis 1 starts at dim 16
        (18, (0, 1, 0), THETA ** (-2.0 / 56)),                 # axis 1, pair 1
        (72, (0, 0, 7), 7.0),                                  # axis 2 starts at dim 72
        (126, (0, 0, 3), 3.0 * THETA ** (-54.0 / 56)),         # last pair of axis 2
        (16, (9, 0, 4), 0.0),                                  # axis 1 untouched by axes 0 and 2
    ]
    for dim, p, ang in cases:
        x = np.zeros((1, 1, 1, D))
        x[..., dim] = 1.0
        got = oracle.prologue(x, np.array([p], np.int32), np.ones(D))[0, 0, 0]
        want = np.zeros(D)
        want[dim] = u * math.cos(ang)
        want[dim + 1] = u * math.sin(ang)
        _close(got, want, 1e-12, "RoPE hand case dim=%d pos=%s" % (dim, p))


def check_rope_pair_norms():
    rng = _rng(6)
    x = rng.standard_normal((1, 7, 2, D))
    w = 1.0 + 0.1 * rng.standard_normal(D)
    pos = rng.integers(0, 300, (7, 3)).astype(np.int32)
    a = oracle.prologue(x, pos, w)
    b = oracle.prologue(x, np.zeros_like(pos), w)
    na = a[..., 0::2] ** 2 + a[..., 1::2] ** 2
    nb = b[..., 0::2] ** 2 + b[..., 1::2] ** 2
    _close(na, nb, 1e-11, "RoPE pair norms")
    assert np.max(np.abs(a - b)) > 1e-3, "RoPE did nothing at nonzero positions"


# ------------------------------------------------------------- attention

def _geometry(txt=5, ih=4, iw=8, rh=0, rw=0):
    return position_ids(txt, ih, iw, rh, rw)


def check_attention_matches_torch_sdpa():
    rng = _rng(7)
    pos = _geometry(5, 4, 8, 2, 3)
    N = pos.shape[0]
    q = rng.standard_normal((2, N, 3, D))
    k = rng.standard_normal((2, N, 3, D))
    v = rng.standard_normal((2, N, 3, D))
    wq = 1.0 + 0.1 * rng.standard_normal(D)
    wk = 1.0 + 0.1 * rng.standard_normal(D)
    got = oracle.attention_rows(q, k, v, pos, wq, wk)
    want = lib_attention(lib_rope(lib_rms(q, wq), pos), lib_rope(lib_rms(k, wk), pos), v)
    _close(got, want, 1e-12, "attention vs torch SDPA")


def check_bf16_entry_matches_f64_entry():
    rng = _rng(8)
    pos = _geometry(3, 3, 5)
    N = pos.shape[0]
    bits = [bf16_bits_from_f32(rng.standard_normal((1, N, 2, D)).astype(np.float32)) for _ in range(3)]
    as64 = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy() for b in bits]
    assert np.array_equal(as64[0], bf16_bits_to_f32(bits[0]).astype(np.float64))
    wq = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    a = oracle.attention_rows(*bits, pos, wq, wk)
    b = oracle.attention_rows(*as64, pos, wq.astype(np.float64), wk.astype(np.float64))
    assert np.array_equal(a, b), "bf16 and fp64 entry points disagree"


def _rand_head(seed, N=23, H=2, B=1):
    rng = _rng(seed)
    pos = rng.integers(0, 40, (N, 3)).astype(np.int32)
    q, k, v = (rng.standard_normal((B, N, H, D)) for _ in range(3))
    wq = 1.0 + 0.1 * rng.standard_normal(D)
    wk = 1.0 + 0.1 * rng.standard_normal(D)
    return q, k, v, pos, wq, wk


def check_softmax_rows_sum_to_one():
    q, k, v, pos, wq, wk = _rand_head(9)
    v[..., 5] = 1.0
    o = oracle.attention_rows(q, k, v, pos, wq, wk)
    _close(o[..., 5], 1.0, 1e-13, "softmax row sum")


def check_constant_v():
    q, k, v, pos, wq, wk = _rand_head(10)
    v[:] = np.linspace(-2, 2, D)
    o = oracle.attention_rows(q, k, v, pos, wq, wk)
    _close(o, v, 1e-13, "constant V")


def check_zero_q_is_mean_v():
    q, k, v, pos, wq, wk = _rand_head(11)
    q[:] = 0.0
    o = oracle.attention_rows(q, k, v, pos, wq, wk)
    want = np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape)
    _close(o, want, 1e-13, "zero Q gives mean of V")


def check_single_token():
    q, k, v, pos, wq, wk = _rand_head(12, N=1, H=3)
    o = oracle.attention_rows(q, k, v, pos, wq, wk)
    _close(o, v, 1e-14, "single token returns v")


def check_permutation_equivariance():
    q, k, v, pos, wq, wk = _rand_head(13, N=29)
    perm = _rng(14).permutation(29)
    o = oracle.attention_rows(q, k, v, pos, wq, wk)
    op = oracle.attention_rows(q[:, perm], k[:, perm], v[:, perm], pos[perm], wq, wk)
    _close(op, o[:, perm], 1e-12, "permutation equivariance")


def check_common_shift_invariance():
    q, k, v, pos, wq, wk = _rand_head(15, N=31)
    o = oracle.attention_rows(q, k, v, pos, wq, wk)
    for axis, delta in ((0, 3), (1, -17), (2, 101)):
        p2 = pos.copy()
        p2[:, axis] += delta
        o2 = oracle.attention_rows(q, k, v, p2, wq, wk)
        _close(o2, o, 1e-11, "shift of axis %d" % axis)
    p3 = pos.copy()
    p3[0, 1] += 5                                   # moving one token does change the output
    assert np.max(np.abs(oracle.attention_rows(q, k, v, p3, wq, wk) - o)) > 1e-6


def check_hand_two_token_head():
    """Two tokens, one head, w = 1, positions zero.
    q_0 = 2 e_0, q_1 = e_1; k_0 = e_0, k_1 = 3 e_1 + 3 e_0 (norm spread over two dims);
    v_0 = e_2, v_1 = e_3."""
    u1 = 1.0 / math.sqrt(1.0 / D + EPS)                 # RMSNorm of a one-hot row (any scale c:
    uc = lambda c: c / math.sqrt(c * c / D + EPS)       #   c / sqrt(c^2/d + eps))
    u2 = 3.0 / math.sqrt(18.0 / D + EPS)                # RMSNorm of 3 e_0 + 3 e_1
    q = np.zeros((1, 2, 1, D)); k = np.zeros((1, 2, 1, D)); v = np.zeros((1, 2, 1, D))
    q[0, 0, 0, 0] = 2.0
    q[0, 1, 0, 1] = 1.0
    k[0, 0, 0, 0] = 1.0
    k[0, 1, 0, 0] = 3.0; k[0, 1, 0, 1] = 3.0
    v[0, 0, 0, 2] = 1.0
    v[0, 1, 0, 3] = 1.0
    # scores / sqrt(d)
    s00 = uc(2.0) * u1 / math.sqrt(D)
    s01 = uc(2.0) * u2 / math.sqrt(D)
    s10 = 0.0
    s11 = u1 * u2 / math.sqrt(D)
    p0 = [math.exp(s00) / (math.exp(s00) + math.exp(s01)), math.exp(s01) / (math.exp(s00) + math.exp(s01))]
    p1 = [math.exp(s10) / (math.exp(s10) + math.exp(s11)), math.exp(s11) / (math.exp(s10) + math.exp(s11))]
    o = oracle.attention_rows(q, k, v, np.zeros((2, 3), np.int32), np.ones(D), np.ones(D))
    want = np.zeros((1, 2, 1, D))
    want[0, 0, 0, 2], want[0, 0, 0, 3] = p0
    want[0, 1, 0, 2], want[0, 1, 0, 3] = p1
    _close(o, want, 1e-14, "hand two-token head")


def check_row_subset_matches_full():
    q, k, v, pos, wq, wk = _rand_head(16, N=19, H=3, B=2)
    full = oracle.attention_rows(q, k, v, pos, wq, wk)
    rows = np.array([[1, 2, 18], [0, 0, 0], [1, 0, 7], [0, 2, 3]], np.int64)
    sub = oracle.attention_rows(q, k, v, pos, wq, wk, rows=rows)
    want = np.stack([full[b, n, h] for b, h, n in rows])
    assert np.array_equal(sub, want)


# ------------------------------------------------------------------- FP8

def _fp8_inputs(seed, N=40, H=2, B=2):
    rng = _rng(seed)
    pos = _geometry(8, 4, 8)
    assert pos.shape[0] == N
    def draw():
        x = rng.standard_normal((B, N, H, D)).astype(np.float32)
        m = rng.random((B, N, H, D)) < 0.01
        x[m] *= 8.0
        return bf16_bits_from_f32(x)
    q, k, v = draw(), draw(), draw()
    wq = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    return q, k, v, pos, wq, wk


def _torch_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn)


def check_fp8_codes_and_scales():
    q, k, v, pos, wq, wk = _fp8_inputs(17)
    qn = oracle.prologue(q, pos, wq)
    kn = oracle.prologue(k, pos, wk)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    for b in range(2):
        for h in range(2):
            q8, k8, v8, sc = oracle.fp8_quantize_head(q, k, v, pos, wq, wk, b, h)
            for name, x, codes, s in (("q", qn, q8, sc[0]), ("k", kn, k8, sc[1]), ("v", vf, v8, sc[2])):
                xs = x[b, :, h, :]
                amax = np.max(np.abs(xs))
                want_s = amax / 448.0
                assert abs(s - want_s) <= 1e-15 * want_s, "%s scale" % name
                want = _torch_e4m3(448.0 * xs / amax).view(torch.uint8).numpy()
                assert np.array_equal(codes, want), "%s codes differ from torch's cast" % name


def check_fp8_codes_at_exact_ties():
    """A quotient x / scale exactly halfway between two E4M3 codes takes the
    even one.  With amax = 30.5, x = 183/2048 gives x / scale = 1.3125,
    halfway between 1.25 (code 58, even mantissa) and 1.375 (code 59);
    x = 183/512 gives 5.25, between 5.0 (code 74) and 5.5 (code 75).  Dividing
    by a rounded scale (x / fl(amax / 448) = 1.3125000000000002) takes 59."""
    q, k, v, pos, wq, wk = _fp8_inputs(20)
    head = np.zeros((v.shape[1], D), np.float32)
    head[0, 0] = 30.5
    head[1, 5] = 183.0 / 2048
    head[2, 7] = -183.0 / 2048
    head[3, 9] = 183.0 / 512
    head[4, 11] = 1.0 / 16        # 0.0625 * 448 / 30.5 = 0.918...: not a tie, rounds to 0.9375 (code 55)
    v[0, :, 0, :] = bf16_bits_from_f32(head)
    _, _, v8, sc = oracle.fp8_quantize_head(q, k, v, pos, wq, wk, 0, 0)
    assert sc[2] == 30.5 / 448.0
    assert v8[0, 0] == 0x7E and v8[1, 5] == 58 and v8[2, 7] == 0x80 | 58 and v8[3, 9] == 74
    assert v8[4, 11] == 55
    assert np.all(v8[5:] == 0)


def check_fp8_attention_on_dequantised_inputs():
    q, k, v, pos, wq, wk = _fp8_inputs(18)
    got = oracle.attention_rows(q, k, v, pos, wq, wk, fp8=True)
    qn = oracle.prologue(q, pos, wq)
    kn = oracle.prologue(k, pos, wk)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    deq = []
    for x in (qn, kn, vf):
        y = np.empty_like(x)
        for b in range(x.shape[0]):
            for h in range(x.shape[2]):
                xs = x[b, :, h, :]
                s = np.max(np.abs(xs)) / 448.0
                y[b, :, h, :] = _torch_e4m3(xs / s).to(torch.float64).numpy() * s
        deq.append(y)
    want = lib_attention(*deq)
    _close(got, want, 1e-12, "FP8 attention vs SDPA on dequantised inputs")
    # and it is not the unquantised result
    plain = oracle.attention_rows(q, k, v, pos, wq, wk)
    assert np.max(np.abs(plain - got)) > 1e-4


def check_fp8_quantize_values_is_the_head_quantiser():
    """The array entry point quantises like the per-head one (reading R5), and
    matches torch's cast of 448 x / amax."""
    q, k, v, pos, wq, wk = _fp8_inputs(25)
    qn = oracle.prologue(q, pos, wq)
    q8, _, v8, sc = oracle.fp8_quantize_head(q, k, v, pos, wq, wk, 1, 0)
    codes, scale = oracle.fp8_quantize(qn[1, :, 0, :])
    assert np.array_equal(codes, q8) and scale == sc[0]
    vf = bf16_bits_to_f32(v).astype(np.float64)[1, :, 0, :]
    codes, scale = oracle.fp8_quantize(vf)
    assert np.array_equal(codes, v8) and scale == sc[2]
    x = np.linspace(-3.0, 5.0, 77)
    codes, scale = oracle.fp8_quantize(x)
    assert scale == 5.0 / 448.0
    assert np.array_equal(codes, _torch_e4m3(448.0 * x / 5.0).view(torch.uint8).numpy())
    codes, scale = oracle.fp8_quantize(np.zeros(5))
    assert scale == 1.0 and not codes.any()


def check_fp8_zero_head():
    q, k, v, pos, wq, wk = _fp8_inputs(19)
    q[:, :, 1] = 0; k[:, :, 1] = 0; v[:, :, 1] = 0
    o = oracle.attention_rows(q, k, v, pos, wq, wk, fp8=True)
    assert np.all(o[:, :, 1] == 0.0)
    _, _, _, sc = oracle.fp8_quantize_head(q, k, v, pos, wq, wk, 0, 1)
    assert np.all(sc == 1.0)


# ------------------------------------------------- VC-Attention repair (R7)

def _lib_deq(x):
    """Dequantised copy of one head's [N, d] values by torch's E4M3 cast (R5)."""
    amax = float(np.max(np.abs(x)))
    if amax == 0.0:
        return x.copy()
    return _torch_e4m3(448.0 * x / amax).to(torch.float64).numpy() * (amax / 448.0)


def _lib_vc(q, k, v, pos, wq, wk, rho):
    """Brute-force VC-Attention from library routines: (output [B, N, H, d],
    per-head errors {(b, h): [N]}, per-head selections {(b, h): sorted list})."""
    qn = lib_rope(lib_rms(bf16_bits_to_f32(q).astype(np.float64), wq), pos)
    kn = lib_rope(lib_rms(bf16_bits_to_f32(k).astype(np.float64), wk), pos)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    B, N, H, _ = q.shape
    R = min(N, max(0, math.ceil(rho * N)))
    qd, kh, vh = np.empty_like(qn), np.empty_like(kn), np.empty_like(vf)
    errs, sels = {}, {}
    for b in range(B):
        for h in range(H):
            qd[b, :, h] = _lib_deq(qn[b, :, h])
            kd, vd = _lib_deq(kn[b, :, h]), _lib_deq(vf[b, :, h])
            err = ((kn[b, :, h] - kd) ** 2).sum(axis=1) + ((vf[b, :, h] - vd) ** 2).sum(axis=1)
            chosen = sorted(sorted(range(N), key=lambda m: (-err[m], m))[:R])
            kd[chosen] = kn[b, chosen, h]
            vd[chosen] = vf[b, chosen, h]
            kh[b, :, h], vh[b, :, h] = kd, vd
            errs[(b, h)], sels[(b, h)] = err, chosen
    return lib_attention(qd, kh, vh), errs, sels


def check_vc_matches_library_reference():
    q, k, v, pos, wq, wk = _fp8_inputs(21)
    for rho in (0.05, 0.3):
        want, errs, sels = _lib_vc(q, k, v, pos, wq, wk, rho)
        got = oracle.vc_attention_rows(q, k, v, pos, wq, wk, rho)
        _close(got, want, 1e-12, "VC rho=%g vs the library reference" % rho)
        assert oracle.vc_repair_count(rho, q.shape[1]) == len(sels[(0, 0)])
        for (b, h), chosen in sels.items():
            sel, err = oracle.vc_select_head(q, k, v, pos, wq, wk, rho, b, h)
            assert list(sel) == chosen, "VC selection of head (%d, %d)" % (b, h)
            np.testing.assert_allclose(err, errs[(b, h)], rtol=1e-10, atol=1e-300)


def check_vc_rho_zero_is_fp8_and_rho_one_exact_kv():
    q, k, v, pos, wq, wk = _fp8_inputs(22)
    plain = oracle.attention_rows(q, k, v, pos, wq, wk, fp8=True)
    assert np.array_equal(oracle.vc_attention_rows(q, k, v, pos, wq, wk, 0.0), plain)
    qn = lib_rope(lib_rms(bf16_bits_to_f32(q).astype(np.float64), wq), pos)
    kn = lib_rope(lib_rms(bf16_bits_to_f32(k).astype(np.float64), wk), pos)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    qd = np.empty_like(qn)
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            qd[b, :, h] = _lib_deq(qn[b, :, h])
    _close(oracle.vc_attention_rows(q, k, v, pos, wq, wk, 1.0), lib_attention(qd, kn, vf), 1e-12,
           "VC rho=1 vs SDPA over dequantised Q' and exact K', V")


def _plant(v, b, h, n, rng):
    """V row n of head (b, h) at +-7 (7 * 448 / 7.75 = 404.6: between the codes
    384 and 416, an error of 11.4 code steps per element) with the head's
    amax 7.75 set elsewhere: by far the head's worst-quantised token."""
    row = np.where(rng.random(D) < 0.5, -7.0, 7.0).astype(np.float32)
    v[b, n, h] = bf16_bits_from_f32(row)
    other = bf16_bits_to_f32(v[b, n - 1, h]).copy()
    other[0] = 7.75
    v[b, n - 1, h] = bf16_bits_from_f32(other)


def check_vc_equal_errors_take_the_lower_index():
    q, k, v, pos, wq, wk = _fp8_inputs(23)
    rng = _rng(23)
    _plant(v, 1, 0, 2, rng)
    k[1, 5, 0], v[1, 5, 0] = k[1, 2, 0], v[1, 2, 0]   # text tokens 2 and 5 share position (0, 0, 0)
    N = q.shape[1]
    sel1, err = oracle.vc_select_head(q, k, v, pos, wq, wk, 0.5 / N, 1, 0)
    assert err[2] == err[5] and err[2] == err.max()
    assert list(sel1) == [2]
    sel2, _ = oracle.vc_select_head(q, k, v, pos, wq, wk, 1.5 / N, 1, 0)
    assert list(sel2) == [2, 5]


def check_vc_planted_token_is_always_repaired():
    q, k, v, pos, wq, wk = _fp8_inputs(24)
    _plant(v, 0, 1, 17, _rng(24))
    N = q.shape[1]
    plain = oracle.attention_rows(q, k, v, pos, wq, wk, fp8=True)
    for rho in (0.5 / N, 0.1, 0.6):
        sel, err = oracle.vc_select_head(q, k, v, pos, wq, wk, rho, 0, 1)
        assert 17 in sel and np.argmax(err) == 17
        assert np.all(np.diff(sel) > 0)
        got = oracle.vc_attention_rows(q, k, v, pos, wq, wk, rho)
        assert np.max(np.abs(got[0, :, 1] - plain[0, :, 1])) > 1e-4   # the repair matters


# ---------------------------------------------------- Sol-Attention (R8)

def _lib_sol_mask(qn, kn, tau):
    """Mask and masses of one head's [N, d] Q', K' from torch routines."""
    N, d = qn.shape
    nb = (N + 127) // 128
    blocks = [slice(128 * j, min(N, 128 * j + 128)) for j in range(nb)]
    qb = torch.stack([torch.from_numpy(qn[b]).mean(0) for b in blocks])
    kb = torch.stack([torch.from_numpy(kn[b]).mean(0) for b in blocks])
    cnt = torch.tensor([b.stop - b.start for b in blocks], dtype=torch.float64)
    mass = torch.softmax(qb @ kb.T / math.sqrt(d) + torch.log(cnt)[None, :], dim=1).numpy()
    keep = mass >= tau / nb
    keep[np.arange(nb), np.argmax(mass, axis=1)] = True
    return keep, mass


def _sol_inputs(seed):
    rng = _rng(seed)
    pos = _geometry(40, 12, 20, 4, 9)        # N = 40 + 240 + 36 = 316: three blocks, the last ragged
    N = pos.shape[0]
    draw = lambda: bf16_bits_from_f32(rng.standard_normal((1, N, 2, D)).astype(np.float32))
    q, k, v = draw(), draw(), draw()
    # give query block 1 a preference: its queries lean toward key block 2
    qf = bf16_bits_to_f32(q).copy()
    kf = bf16_bits_to_f32(k).copy()
    dirn = rng.standard_normal(D).astype(np.float32)
    qf[0, 128:256, 0] += 3.0 * dirn
    kf[0, 256:, 0] += 3.0 * dirn
    q, k = bf16_bits_from_f32(qf), bf16_bits_from_f32(kf)
    wq = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    return q, k, v, pos, wq, wk


def check_sol_mask_matches_library():
    q, k, v, pos, wq, wk = _sol_inputs(31)
    qn = lib_rope(lib_rms(bf16_bits_to_f32(q).astype(np.float64), wq), pos)
    kn = lib_rope(lib_rms(bf16_bits_to_f32(k).astype(np.float64), wk), pos)
    for tau in (0.5, 1.0, 1.6):
        for h in range(2):
            keep, mass = oracle.sol_mask(q, k, pos, wq, wk, tau, 0, h)
            want_keep, want_mass = _lib_sol_mask(qn[0, :, h], kn[0, :, h], tau)
            _close(mass, want_mass, 1e-12, "Sol block masses, head %d" % h)
            assert np.array_equal(keep, want_keep), ("Sol mask", tau, h, keep, want_keep)
    keep, mass = oracle.sol_mask(q, k, pos, wq, wk, 1.0, 0, 0)
    assert keep[1, 2] and mass[1, 2] > 0.5          # the planted preference
    _close(mass.sum(axis=1), np.ones(3), 1e-12, "Sol masses sum to one")


def check_sol_tau_zero_is_dense():
    q, k, v, pos, wq, wk = _sol_inputs(32)
    dense = oracle.attention_rows(q, k, v, pos, wq, wk)
    _close(oracle.sol_attention_rows(q, k, v, pos, wq, wk, 0.0), dense, 1e-14, "Sol tau=0 vs dense")


def check_sol_one_block_is_subset_attention():
    """A tau above nb leaves only each query block's block of largest mass:
    the rows are SDPA over that block's keys alone."""
    q, k, v, pos, wq, wk = _sol_inputs(33)
    qn = lib_rope(lib_rms(bf16_bits_to_f32(q).astype(np.float64), wq), pos)
    kn = lib_rope(lib_rms(bf16_bits_to_f32(k).astype(np.float64), wk), pos)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    got = oracle.sol_attention_rows(q, k, v, pos, wq, wk, 10.0)
    N = pos.shape[0]
    for h in range(2):
        keep, _ = _lib_sol_mask(qn[0, :, h], kn[0, :, h], 10.0)
        for i in range(keep.shape[0]):
            (j,) = np.nonzero(keep[i])[0]
            qs, ks = slice(128 * i, min(N, 128 * i + 128)), slice(128 * j, min(N, 128 * j + 128))
            want = lib_attention(qn[:, qs, h:h + 1], kn[:, ks, h:h + 1], vf[:, ks, h:h + 1])
            _close(got[:, qs, h:h + 1], want, 1e-12, "Sol one block, head %d, query block %d" % (h, i))


# --------------------------------------------------------- QKV projection

def _bf16(a):
    bits = bf16_bits_from_f32(np.asarray(a, np.float32))
    return bits, bf16_bits_to_f32(bits).astype(np.float64)


def check_qkv_matches_numpy_matmul():
    """x W^T + b by numpy in fp64, split into Q, K, V heads; Q and K through
    torch rms_norm and the complex-rotation RoPE."""
    rng = _rng(21)
    B, N, H, Dm = 2, 5, 2, 96
    pos = rng.integers(0, 30, (N, 3)).astype(np.int32)
    xb, x = _bf16(rng.standard_normal((B * N, Dm)))
    wb, w = _bf16(rng.standard_normal((3 * H * D, Dm)) / 8)
    bias = rng.standard_normal(3 * H * D).astype(np.float32)
    wq = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    q, k, v = oracle.qkv_rows(xb, wb, bias, N, pos, wq, wk, H)
    y = x @ w.T + bias.astype(np.float64)
    parts = [y[:, i * H * D:(i + 1) * H * D].reshape(B, N, H, D) for i in range(3)]
    want_q = lib_rope(lib_rms(parts[0], wq.astype(np.float64)), pos).reshape(B * N, H, D)
    want_k = lib_rope(lib_rms(parts[1], wk.astype(np.float64)), pos).reshape(B * N, H, D)
    _close(q, want_q, 1e-11, "QKV: Q vs numpy matmul + torch rms_norm + rotation")
    _close(k, want_k, 1e-11, "QKV: K vs numpy matmul + torch rms_norm + rotation")
    _close(v, parts[2].reshape(B * N, H, D), 1e-12, "QKV: V vs numpy matmul")


def check_qkv_identity_weights():
    """W_q = I, W_k = 2 I, W_v = I (D = H d), no bias: Q' is the prologue of x,
    V is x."""
    rng = _rng(22)
    N, H = 7, 2
    Dm = H * D
    pos = _geometry(1, 2, 3)
    xb, x = _bf16(rng.standard_normal((N, Dm)))
    eye = np.eye(Dm)
    wb, _ = _bf16(np.concatenate([eye, 2 * eye, eye], 0))
    ones = np.ones(D, np.float32)
    q, k, v = oracle.qkv_rows(xb, wb, None, N, pos, ones, ones, H)
    xh = x.reshape(1, N, H, D)
    _close(q, oracle.prologue(xh, pos, np.ones(D))[0], 1e-12, "QKV identity: Q")
    _close(k, oracle.prologue(2 * xh, pos, np.ones(D))[0], 1e-12, "QKV identity: K")
    _close(v, xh[0], 0.0, "QKV identity: V")


def check_qkv_bias_only():
    """W = 0: every token's V is the V part of the bias, Q' and K' the
    normalised, rotated bias parts."""
    rng = _rng(23)
    N, H, Dm = 4, 3, 32
    pos = _geometry(2, 1, 2)
    xb, _ = _bf16(rng.standard_normal((N, Dm)))
    wb, _ = _bf16(np.zeros((3 * H * D, Dm)))
    bias = rng.standard_normal(3 * H * D).astype(np.float32)
    ones = np.ones(D, np.float32)
    q, k, v = oracle.qkv_rows(xb, wb, bias, N, pos, ones, ones, H)
    bq, bk, bv = (bias.astype(np.float64)[i * H * D:(i + 1) * H * D].reshape(H, D) for i in range(3))
    _close(v, np.broadcast_to(bv, (N, H, D)), 0.0, "QKV bias only: V")
    bqn = np.broadcast_to(bq, (1, N, H, D)).copy()
    _close(q, lib_rope(lib_rms(bqn, np.ones(D)), pos)[0], 1e-12, "QKV bias only: Q")
    _close(k, lib_rope(lib_rms(np.broadcast_to(bk, (1, N, H, D)).copy(), np.ones(D)), pos)[0], 1e-12,
           "QKV bias only: K")


ALL_CHECKS = [
    check_e4m3_exhaustive_roundtrip,
    check_e4m3_matches_torch_cast,
    check_e4m3_ties_and_saturation,
    check_rmsnorm_matches_torch,
    check_rmsnorm_closed_form,
    check_rope_complex_form,
    check_rope_hand_cases,
    check_rope_pair_norms,
    check_attention_matches_torch_sdpa,
    check_bf16_entry_matches_f64_entry,
    check_softmax_rows_sum_to_one,
    check_constant_v,
    check_zero_q_is_mean_v,
    check_single_token,
    check_permutation_equivariance,
    check_common_shift_invariance,
    check_hand_two_token_head,
    check_row_subset_matches_full,
    check_fp8_codes_and_scales,
    check_fp8_attention_on_dequantised_inputs,
    check_fp8_zero_head,
    check_fp8_quantize_values_is_the_head_quantiser,
    check_fp8_codes_at_exact_ties,
    check_qkv_matches_numpy_matmul,
    check_qkv_identity_weights,
    check_qkv_bias_only,
    check_vc_matches_library_reference,
    check_vc_rho_zero_is_fp8_and_rho_one_exact_kv,
    check_vc_equal_errors_take_the_lower_index,
    check_vc_planted_token_is_always_repaired,
    check_sol_mask_matches_library,
    check_sol_tau_zero_is_dense,
    check_sol_one_block_is_subset_attention,
]
