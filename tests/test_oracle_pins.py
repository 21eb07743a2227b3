"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle step to a closed form, an exhaustive enumeration, a
library routine, an invariant, a hand-worked example or an independent brute
force, so that a dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import mx_ref
import synth

E4M3, E2M1 = oracle.FMT_E4M3, oracle.FMT_E2M1
FMT = {"E4M3": E4M3, "E2M1": E2M1}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_hand_examples.txt")


# --------------------------------------------------------------------------
# codebooks
# --------------------------------------------------------------------------

def test_e4m3_codebook_matches_torch_float8():
    """Every E4M3 code decodes to torch's float8_e4m3fn value (NaN at 0x7F/0xFF)."""
    ref = mx_ref.e4m3_decode_all()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e2m1_codebook_and_e8m0():
    assert [oracle.e2m1_decode(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for c in range(8):
        v = oracle.e2m1_decode(c + 8)
        assert v == -oracle.e2m1_decode(c) and math.copysign(1, v) == -1
    for s in range(255):
        assert oracle.e8m0_decode(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(oracle.e8m0_decode(255))


@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_codebook_round_trip(fmt):
    """encode(decode(c)) == c for every non-NaN code, including the signed zero."""
    n = 256 if fmt == E4M3 else 16
    for c in range(n):
        v = oracle.e4m3_decode(c) if fmt == E4M3 else oracle.e2m1_decode(c)
        if math.isnan(v):
            continue
        assert oracle.mx_encode(v, fmt) == c, (fmt, hex(c), v)


def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = mx_ref.bf16_bits_to_f64(bits)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_encode_matches_arithmetic_rne_on_every_bf16(fmt):
    """Codebook search == arithmetic round-half-even (frexp) on all finite bf16 values."""
    v = _all_bf16_values()
    codes = np.array([oracle.mx_encode(float(y), fmt) for y in v])
    got = mx_ref.decode(codes, fmt)
    want = mx_ref.rne_value(v, fmt)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(v))  # sign kept, also on zeros


def test_e4m3_encode_matches_torch_cast_in_range():
    """Inside the finite range torch's RNE cast to float8_e4m3fn agrees code for code."""
    v = _all_bf16_values()
    v = v[np.abs(v) <= 448.0]
    want = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.mx_encode(float(y), E4M3) for y in v], dtype=np.uint8)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_decode_encode_within_half_quantum(fmt):
    v = _all_bf16_values()
    maxv = mx_ref.MAXV[fmt]
    v = v[np.abs(v) <= maxv]
    codes = np.array([oracle.mx_encode(float(y), fmt) for y in v])
    d = mx_ref.decode(codes, fmt)
    _, ex = np.frexp(np.where(v != 0, np.abs(v), 1.0))
    q = np.ldexp(1.0, np.maximum(ex - 1, mx_ref.EMIN[fmt]) - mx_ref.MBITS[fmt])
    assert np.all(np.abs(d - v) <= q / 2)


# --------------------------------------------------------------------------
# scale rule
# --------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_scale_closed_form_over_every_binade(fmt):
    """amax = m * 2^p -> scale byte clamp(p - emax + 127, 0, 254), for every normal binade."""
    emax = mx_ref.EMAX[fmt]
    for p in range(-126, 128):
        for m in (1.0, 1.25, 1.5, 1.999):
            amax = np.float32(math.ldexp(m, p))
            if not np.isfinite(amax):
                continue
            s = oracle.mx_scale_byte(float(amax), fmt)
            assert s == min(max(p - emax + 127, 0), 254), (p, m, s)
    assert oracle.mx_scale_byte(0.0, fmt) == 0
    assert oracle.mx_scale_byte(float(np.float32(1e-40)), fmt) == 0  # subnormal


@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_block_property_largest_element_lands_in_top_binade(fmt):
    """After dividing by X the block's largest magnitude lies in [2^emax, 2^(emax+1)),
    so its code is either in the format's top binade or saturated to max."""
    rng = np.random.default_rng(7)
    emax = mx_ref.EMAX[fmt]
    for _ in range(500):
        v = (rng.standard_normal(32) * np.exp(rng.uniform(-30, 30))).astype(np.float32)
        codes, s = oracle.quantize_block(v, fmt)
        X = math.ldexp(1.0, s - 127)
        a = float(np.abs(v).max()) / X
        assert 2.0 ** emax <= a < 2.0 ** (emax + 1)
        i = int(np.abs(v).argmax())
        dv = abs(mx_ref.decode(codes[i], fmt))
        assert dv >= 2.0 ** emax


def _parse_code(tok):
    return None if tok == "none" else int(tok, 16)


def test_hand_worked_examples():
    nblock = nenc = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "block":
                _, fmt, fill, nfill, other, sbyte, cfill, cother = parts
                v = np.full(32, float(other), np.float32)
                v[: int(nfill)] = float(fill)
                codes, s = oracle.quantize_block(v, FMT[fmt])
                assert s == int(sbyte), line
                assert codes[0] == _parse_code(cfill), line
                if _parse_code(cother) is not None:
                    assert codes[31] == _parse_code(cother), line
                nblock += 1
            elif parts[0] == "encode":
                _, fmt, val, code = parts
                assert oracle.mx_encode(float(val), FMT[fmt]) == int(code, 16), line
                nenc += 1
    assert nblock >= 7 and nenc >= 20


@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_quantize_rows_matches_independent_reference(fmt):
    """Row quantiser (codes, nibble packing, scale layout) vs the numpy restatement."""
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((9, 256)) * rng.uniform(1e-3, 1e3, (9, 1))).astype(np.float32)
    v[4, 32:64] = 0.0  # an all-zero block
    v[5, :32] *= 1e-38  # a block whose amax is fp32-subnormal
    codes, scales = oracle.quantize_rows_f32(v, fmt)
    want_vals, want_sc = mx_ref.quantize_values(v, fmt)
    assert np.array_equal(scales, want_sc)
    if fmt == E2M1:
        codes = mx_ref.unpack_fp4(codes)
    got_vals = mx_ref.decode(codes, fmt) * np.repeat(np.ldexp(1.0, scales.astype(int) - 127), 32, axis=1)
    assert np.array_equal(got_vals, want_vals)
    assert np.array_equal(np.signbit(got_vals), np.signbit(want_vals))


@pytest.mark.parametrize("fmt", [E4M3, E2M1])
def test_dequantize_rows_against_torch_and_tables(fmt):
    """Row decoder: every code (E4M3 through torch's float8_e4m3fn, E2M1 through the literal
    table with element 2i in the low nibble) times 2^(s - 127) of its 32-block's scale byte."""
    rng = np.random.default_rng(17)
    rows, K = 5, 256
    if fmt == E4M3:
        codes = rng.integers(0, 256, (rows, K), dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes: the quantiser never emits them
        elem = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    else:
        codes = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
        table = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                          -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
        elem = np.empty((rows, K))
        elem[:, 0::2] = table[codes & 15]
        elem[:, 1::2] = table[codes >> 4]
    scales = rng.integers(0, 255, (rows, K // 32), dtype=np.uint8)
    scales[0, 0], scales[1, 1] = 0, 254  # the extreme finite scales
    got = oracle.dequantize_rows(codes, scales, K, fmt)
    want = elem * np.ldexp(1.0, np.repeat(scales.astype(int), 32, axis=1) - 127)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    # and it inverts the row quantiser on values that lie on the MX grid
    v = (elem[:2] * 2.0 ** -3).astype(np.float32)
    c, sc = oracle.quantize_rows_f32(v, fmt)
    back = oracle.dequantize_rows(c, sc, K, fmt)
    assert np.array_equal(back, v.astype(np.float64))


def test_bf16_rows_and_nibble_order():
    """bf16 entry point equals the fp32 one; FP4 element 2i sits in the low nibble."""
    x = synth.x_bf16(4, 128, seed=11)
    bits = synth.bf16_bits(x)
    c1, s1 = oracle.quantize_rows_bf16(bits, E2M1)
    c2, s2 = oracle.quantize_rows_f32(x.float().numpy(), E2M1)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    v = np.zeros((1, 32), np.float32)
    v[0, 0] = 6.0  # code 7, element 0 -> low nibble of byte 0
    v[0, 3] = -1.0  # code 0xA, element 3 -> high nibble of byte 1
    c, s = oracle.quantize_rows_f32(v, E2M1)
    assert s[0, 0] == 127 and c[0, 0] == 0x07 and c[0, 1] == 0xA0


def test_bf16_output_rounding():
    rng = np.random.default_rng(5)
    d = rng.standard_normal(4000) * np.exp(rng.uniform(-80, 80, 4000))
    d = np.concatenate([d, [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0]])
    got = mx_ref.bf16_bits_to_f64(np.array([oracle.f64_to_bf16(float(v)) for v in d], np.uint16))
    want = mx_ref.bf16_rne(d)
    assert np.array_equal(got, want)
    assert got[-5] == 1.0 and got[-4] == 1.0 + 2 ** -6  # ties to even


# --------------------------------------------------------------------------
# routing and permutation
# --------------------------------------------------------------------------

def test_route_brute_force_and_invariants():
    E, k = 64, 6
    lg = synth.gate_logits(300, E, seed=2).numpy()
    lg[0, :] = 0.5  # all tied: must pick experts 0..k-1
    lg[1, 10] = lg[1, 3] = 9.0  # two tied maxima
    ids, w = oracle.route(lg, k)
    for t in range(lg.shape[0]):
        order = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
        assert list(ids[t]) == order
        assert len(set(ids[t])) == k
        assert np.all(np.diff(lg[t, ids[t]]) <= 0)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) <= k * 2.0 ** -23
        assert np.all(np.diff(w[t]) <= 1e-7)
        p = torch.softmax(torch.from_numpy(lg[t]).double(), 0).numpy()[ids[t]]
        assert np.allclose(w[t], p / p.sum(), rtol=1e-6, atol=0)
    assert list(ids[0]) == list(range(k))
    assert list(ids[1][:2]) == [3, 10]


def test_route_k1_weight_is_one():
    lg = synth.gate_logits(50, 16, seed=9).numpy()
    ids, w = oracle.route(lg, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(ids[:, 0], lg.argmax(1))


def test_sort_is_stable_bijection():
    E, k = 37, 3
    lg = synth.gate_logits(500, E, seed=4, skew=True).numpy()
    ids, _ = oracle.route(lg, k)
    counts, offsets, sp, inv = oracle.sort(ids, E)
    R = ids.size
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == R and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(sp), np.arange(R))
    assert np.array_equal(inv[sp], np.arange(R))
    flat = ids.ravel()
    for e in range(E):
        seg = sp[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    assert offsets.dtype == np.int64


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------

def _tiny_case(T=16, H=256, I=128, E=8, k=2, seed=0, act=E4M3):
    x = synth.x_bf16(T, H, seed)
    lg = synth.gate_logits(T, E, seed).numpy()
    w1b, w2b = synth.weights_bf16(E, H, I, seed)
    w1, w1s = oracle.quantize_rows_bf16(synth.bf16_bits(w1b).reshape(E * 2 * I, H), E2M1)
    w2, w2s = oracle.quantize_rows_bf16(synth.bf16_bits(w2b).reshape(E * H, I), E2M1)
    return dict(x=synth.bf16_bits(x), lg=lg, w1=w1.reshape(E, 2 * I, H // 2), w1s=w1s.reshape(E, 2 * I, H // 32),
                w2=w2.reshape(E, H, I // 2), w2s=w2s.reshape(E, H, I // 32), T=T, H=H, I=I, E=E, k=k, act=act,
                w1b=w1b, w2b=w2b)


def _dense_masked(c, h_bf16=False, y2_fp8=False):
    """Brute force over ALL experts for every token, masked by the routing:
    no sort, no gather, numpy matmuls, the numpy MX restatement, torch softmax.
    h_bf16: h rounded to bf16 (numpy round-to-nearest-even) before its quantisation.
    y2_fp8: each expert's rows weighted in fp32 (the routing weights, pinned above) and
    passed through the numpy E4M3 restatement before they are summed."""
    T, H, I, E, k, act = c["T"], c["H"], c["I"], c["E"], c["k"], c["act"]
    x = mx_ref.bf16_bits_to_f64(c["x"]).astype(np.float32)
    xq, _ = mx_ref.quantize_values(x, act)
    W1 = mx_ref.dequant_weights(c["w1"], c["w1s"])  # [E, 2I, H]
    W2 = mx_ref.dequant_weights(c["w2"], c["w2s"])  # [E, H, I]
    lg = torch.from_numpy(c["lg"]).double()
    p = torch.softmax(lg, 1).numpy()
    mask = np.zeros((T, E))
    for t in range(T):
        top = sorted(range(E), key=lambda e: (-float(c["lg"][t, e]), e))[:k]
        mask[t, top] = p[t, top] / p[t, top].sum()
    wmask = np.zeros((T, E), np.float32)  # the fp32 routing weights the layer applies
    if y2_fp8:
        ids, w = oracle.route(c["lg"], k)
        for t in range(T):
            wmask[t, ids[t]] = w[t]
    out = np.zeros((T, H))
    for e in range(E):
        acc = (xq @ W1[e].T).astype(np.float32)  # [T, 2I]
        g, u = acc[:, 0::2], acc[:, 1::2]
        h = (g / (np.float32(1) + np.exp(-g)) * u).astype(np.float32)
        if h_bf16:
            h = mx_ref.bf16_rne(h.astype(np.float64)).astype(np.float32)
        a2, _ = mx_ref.quantize_values(h, act)
        y2 = (a2 @ W2[e].T).astype(np.float32).astype(np.float64)
        if y2_fp8:
            v = wmask[:, e:e + 1] * y2.astype(np.float32)  # fp32 product
            q, _ = mx_ref.quantize_values(v, E4M3)
            out += q
        else:
            out += mask[:, e:e + 1].astype(np.float32).astype(np.float64) * y2
    return out


@pytest.mark.parametrize("h_bf16", [False, True])
@pytest.mark.parametrize("act", [E4M3, E2M1])
def test_forward_equals_dense_masked_brute_force(act, h_bf16):
    c = _tiny_case(act=act)
    got = mx_ref.bf16_bits_to_f64(oracle.moe_forward(c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"],
                                                     c["E"], c["k"], act, h_bf16=h_bf16))
    want = _dense_masked(c, h_bf16)
    ulp = np.ldexp(1.0, np.frexp(np.abs(want) + 1e-30)[1] - 8)
    assert np.all(np.abs(got - want) <= ulp), np.abs(got - want).max()


@pytest.mark.parametrize("act", [E4M3, E2M1])
def test_y2_fp8_option_equals_dense_masked_brute_force(act):
    """FP8 transport of the stage-2 rows ("add A4W4 and FP8 P2P transport support to MegaMoE",
    Technical Details): the weighted rows quantised to E4M3 with one E8M0 scale per 1x32 block
    before the combine.  The brute force builds it from the numpy MX restatement and the pinned
    routing weights; the option moves the output by E4M3 rounding (a few percent), no more."""
    c = _tiny_case(act=act)
    args = (c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], c["k"], act)
    got = mx_ref.bf16_bits_to_f64(oracle.moe_forward(*args, y2_fp8=True))
    want = _dense_masked(c, y2_fp8=True)
    ulp = np.ldexp(1.0, np.frexp(np.abs(want) + 1e-30)[1] - 8)
    assert np.all(np.abs(got - want) <= ulp), np.abs(got - want).max()
    base = mx_ref.bf16_bits_to_f64(oracle.moe_forward(*args))
    rel = np.linalg.norm(got - base) / np.linalg.norm(base)
    assert 1e-3 < rel < 0.1, rel


@pytest.mark.parametrize("act", [E4M3, E2M1])
def test_h_bf16_option_rounds_h_and_requantises_it(act):
    """With h rounded to bf16, the diagnostics' h is the fp32 run's h rounded to nearest even,
    and A2 is the oracle's row quantiser applied to that h; the output moves by the re-rounding
    of a few percent of the A2 codes (a code step across a rounding boundary)."""
    c = _tiny_case(act=act)
    args = (c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], c["k"], act)
    out32, d32 = oracle.moe_forward(*args, diagnostics=True)
    out16, d16 = oracle.moe_forward(*args, diagnostics=True, h_bf16=True)
    assert np.array_equal(d16["h"], mx_ref.bf16_rne(d32["h"].astype(np.float64)).astype(np.float32))
    codes, scales = oracle.quantize_rows_f32(d16["h"].reshape(-1, c["I"]), act)
    assert np.array_equal(codes.reshape(d16["a2"].shape), d16["a2"])
    assert np.array_equal(scales.reshape(d16["a2s"].shape), d16["a2s"])
    a, b = mx_ref.bf16_bits_to_f64(out16), mx_ref.bf16_bits_to_f64(out32)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 0 < rel < 0.1, rel


def test_forward_token_subset_equals_full_rows():
    c = _tiny_case()
    full = oracle.moe_forward(c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], c["k"], E4M3)
    sub = oracle.moe_forward(c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], c["k"], E4M3,
                             tokens=[5, 0, 15])
    assert np.array_equal(sub, full[[5, 0, 15]])


def test_forward_stages_against_fp64_matmul():
    """Each stage of the oracle vs a dense fp64 matmul on the oracle's own intermediates:
    GEMM1+SwiGLU, GEMM2 and the combine are each pinned separately."""
    c = _tiny_case(T=8)
    out, d = oracle.moe_forward(c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], c["k"], E4M3,
                                diagnostics=True)
    ids, w = oracle.route(c["lg"], c["k"])
    x = mx_ref.bf16_bits_to_f64(c["x"]).astype(np.float32)
    xq, _ = mx_ref.quantize_values(x, E4M3)
    W1 = mx_ref.dequant_weights(c["w1"], c["w1s"])
    W2 = mx_ref.dequant_weights(c["w2"], c["w2s"])
    for t in range(c["T"]):
        acc_out = np.zeros(c["H"])
        for j in range(c["k"]):
            e = ids[t, j]
            acc = (W1[e] @ xq[t]).astype(np.float32)
            h = acc[0::2] / (np.float32(1) + np.exp(-acc[0::2])) * acc[1::2]
            assert np.allclose(d["h"][t, j], h, rtol=4e-7, atol=1e-30)
            a2 = mx_ref.decode(d["a2"][t, j], E4M3) * np.repeat(np.ldexp(1.0, d["a2s"][t, j].astype(int) - 127), 32)
            y2 = (W2[e] @ a2).astype(np.float32)
            assert np.array_equal(d["y2"][t, j], y2)
            acc_out += np.float64(w[t, j]) * y2.astype(np.float64)
        assert np.array_equal(mx_ref.bf16_bits_to_f64(out[t]), mx_ref.bf16_rne(acc_out))


def test_forward_special_cases():
    c = _tiny_case()
    zero = np.zeros_like(c["x"])
    out = oracle.moe_forward(zero, c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], c["k"], E4M3)
    assert np.all(mx_ref.bf16_bits_to_f64(out) == 0.0)
    # k = 1: the output is the chosen expert's fp32 GEMM2 row rounded to bf16
    out1, d1 = oracle.moe_forward(c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"], c["E"], 1, E4M3,
                                  diagnostics=True)
    assert np.array_equal(mx_ref.bf16_bits_to_f64(out1), mx_ref.bf16_rne(d1["y2"][:, 0, :].astype(np.float64)))


@pytest.mark.parametrize("act,lo,hi", [(E4M3, 0.005, 0.08), (E2M1, 0.05, 0.3)])
def test_quantisation_error_band(act, lo, hi):
    """Against an unquantised fp64 layer (bf16 x, fp32 h, no activation quantisation) the
    A8W4 error is a few per cent and the A4W4 error roughly ten; a layout or scale bug
    (for instance gate/up mispaired) lands far outside."""
    c = _tiny_case(T=16, act=act)
    got = mx_ref.bf16_bits_to_f64(oracle.moe_forward(c["x"], c["lg"], c["w1"], c["w1s"], c["w2"], c["w2s"],
                                                     c["E"], c["k"], act))
    x = mx_ref.bf16_bits_to_f64(c["x"])
    W1 = mx_ref.dequant_weights(c["w1"], c["w1s"])
    W2 = mx_ref.dequant_weights(c["w2"], c["w2s"])
    ids, w = oracle.route(c["lg"], c["k"])
    ref = np.zeros_like(got)
    for t in range(c["T"]):
        for j in range(c["k"]):
            a = W1[ids[t, j]] @ x[t]
            h = a[0::2] / (1 + np.exp(-a[0::2])) * a[1::2]
            ref[t] += w[t, j] * (W2[ids[t, j]] @ h)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert lo <= rel <= hi, rel
    # the same weights read with gate/up separated instead of interleaved: far off
    E, I, H = c["E"], c["I"], c["H"]
    sep = lambda a: np.concatenate([a[:, 0::2], a[:, 1::2]], axis=1)  # noqa: E731
    bad = mx_ref.bf16_bits_to_f64(oracle.moe_forward(c["x"], c["lg"], sep(c["w1"]), sep(c["w1s"]), c["w2"],
                                                     c["w2s"], E, c["k"], act))
    assert np.linalg.norm(bad - ref) / np.linalg.norm(ref) > 0.5
