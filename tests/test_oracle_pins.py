"""Pins for the CPU oracle: facts the pages and the mathematics fix, checked without
trusting the oracle's own formulas.  CPU only.

Each test names the passage it pins.  Pages: [minfer] "10 . CPU matmul: quantized
weights x Q8_0 activations"; [ggml] "ggml Q4_0 vec_dot Walkthrough"; [krafla]
"Architecture"; [kvad] "kvad -- the same ideas, at scale".
"""
import numpy as np
import pytest

from conftest import read_golden
import workloads

QTYPES = ["q4_0", "q8_0", "q4_K", "q6_K", "q2_K", "q4_1", "q5_0", "q5_1", "q5_K"]
KQUANTS = ("q4_K", "q6_K", "q2_K", "q5_K")


def f16(v):
    return np.float16(v).view(np.uint16).item()


# --------------------------------------------------------------------------- fp16
def test_f16_encode_matches_numpy(orc):
    """The stored scale is IEEE binary16, round to nearest even ([minfer] s3.2, "f16(d)").
    numpy's float32 -> float16 cast is that conversion: compare on random values spanning
    the normal, subnormal, overflow and tie cases."""
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 6, 20000),
        (g.integers(0, 1 << 11, 4000) * 2.0 ** -25).astype(np.float32),        # subnormal ties
        (np.arange(2048, 4096, dtype=np.float32) + np.float32(0.5)),          # ties above 2048
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 2.0 ** -26, 6.1e-5, np.inf, -np.inf], dtype=np.float32),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16_bits(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_f16_decode_all_patterns(orc):
    """binary16 -> binary32 is exact: every one of the 65536 patterns (NaNs by class)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_bits_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# --------------------------------------------------------------------------- formats
def test_block_sizes(orc):
    for row in read_golden("block_sizes.txt"):
        if row[0] == "row":
            assert orc.row_bytes(row[1], int(row[2])) == int(row[3])
        else:
            assert orc.block_bytes(row[0]) == int(row[1])
            assert orc.block_values(row[0]) == int(row[2])


def test_pairing_rule(orc):
    """[minfer] s2.4/s3.2: K-quant weights pair with Q8_K (the Q4_K/Q5_K/Q6_K arms call
    dot_q*_k_q8_k), the 32-value types with Q8_0 (dot_<T>_q8_0)."""
    for t in ("q4_0", "q8_0", "q4_1", "q5_0", "q5_1"):
        assert orc.act_type(t) == orc.Q8_0, t
    for t in KQUANTS:
        assert orc.act_type(t) == orc.Q8_K, t


def _q4_0_block(d_bits, qs):
    return np.array([d_bits & 0xFF, d_bits >> 8] + list(qs), dtype=np.uint8)


def _q8_0_block(d_bits, q):
    return np.array([d_bits & 0xFF, d_bits >> 8] + [int(v) & 0xFF for v in q], dtype=np.uint8)


def test_q4_0_worked_byte(orc):
    """[minfer] s3.2 worked example: byte 0x21 with dx = dy = 1 gives -7 and -6; [ggml] s2:
    byte j holds elements j (low) and j+16 (high).  Checked through both the decoder and
    the integer dot (a one-hot activation picks out a single weight)."""
    for byte, j, lo, hi in read_golden("q4_0_worked_byte.txt"):
        byte, j, lo, hi = int(byte, 16), int(j), int(lo), int(hi)
        qs = [0x88] * 16
        qs[j] = byte
        wb = _q4_0_block(f16(1.0), qs)
        vals = orc.dequantize("q4_0", wb, 32)[0]
        assert vals[j] == lo and vals[j + 16] == hi
        assert np.count_nonzero(vals) == (lo != 0) + (hi != 0)
        for pos, want in ((j, lo), (j + 16, hi)):
            a = [0] * 32
            a[pos] = 1
            xb = _q8_0_block(f16(1.0), a)
            assert orc.blocksums("q4_0", wb, xb, 1, 1, 32)[0, 0, 0] == want
            assert orc.dot_row("q4_0", wb, xb, 32) == float(want)


def test_q4_0_max_magnitude_and_clip(orc):
    """[ggml] s1.1 + [kvad] "The scale that wasted a code": the signed extreme decodes as
    code -8 exactly; the opposite extreme clips to 7/8 of its value."""
    x = np.zeros(32, dtype=np.float32)
    rows = read_golden("q4_0_clip.txt")
    for i, v, _, _ in rows:
        x[int(i)] = float(v)
    q = orc.quantize("q4_0", x)[0]
    vals = orc.dequantize("q4_0", q, 32)[0]
    for i, v, nib, dec in rows:
        i = int(i)
        nibble = (q[2 + i] & 15) if i < 16 else (q[2 + i - 16] >> 4)
        assert nibble == int(nib)
        assert vals[i] == float(dec)


def test_q4_0_quantizer_properties(orc):
    """On random blocks: every code in range, the max-magnitude element at code -8 (decoded
    within the f16 rounding of d), the others within half a step except a clipped extreme."""
    x = workloads.activations_f32(64, 256, seed=7)
    q = orc.quantize("q4_0", x)
    vals = orc.dequantize("q4_0", q, 256)
    codes = orc.codes("q4_0", q, 256)
    assert codes.min() >= -8 and codes.max() <= 7
    xb = x.reshape(-1, 32).astype(np.float64)
    vb = vals.reshape(-1, 32)
    cb = codes.reshape(-1, 32)
    dh = q.reshape(-1)[np.arange(0, q.size, 18)[:, None] + [0, 1]].copy().view(np.uint16).astype(np.float16)
    dh = dh.astype(np.float64).reshape(-1)
    imax = np.abs(xb).argmax(axis=1)
    r = np.arange(xb.shape[0])
    assert np.all(cb[r, imax] == -8)
    m = xb[r, imax]
    d32 = (m / -8.0)
    assert np.all(np.abs(vb[r, imax] - m) <= 8 * np.abs(dh - d32) + 1e-12)
    err = np.abs(vb - xb)
    t = xb / d32[:, None]                      # the code each value wants, before clipping
    unclipped = t < 7.5
    bound = 0.5 * np.abs(dh)[:, None] + np.abs(t) * np.abs(dh - d32)[:, None] + 1e-6 * np.abs(xb)
    assert np.all(err[unclipped] <= bound[unclipped])


def test_q4_0_statistical_pin(orc):
    """[kvad] "The scale that wasted a code": over random blocks the /-8 scale gives a mean
    relative error of 8.49% against 9.54% for the symmetric max/7 scale.  The page does not
    state its distribution or error measure; with N(0,1) blocks of 32 and the per-block
    ratio |x_hat - x| / |x| (L2), the oracle's quantizer reproduces both figures to within
    0.15 points, so the gate is +-0.5 points around the page's numbers."""
    x = np.random.default_rng(3).standard_normal((4096, 32)).astype(np.float32)
    q = orc.quantize("q4_0", x)
    v8 = orc.dequantize("q4_0", q, x.size).reshape(-1, 32)
    amax = np.abs(x).max(axis=1, keepdims=True).astype(np.float64)
    d7 = amax / 7.0
    v7 = np.clip(np.round(x / d7), -8, 7) * d7
    rel8 = np.mean(np.linalg.norm(v8 - x, axis=1) / np.linalg.norm(x, axis=1))
    rel7 = np.mean(np.linalg.norm(v7 - x, axis=1) / np.linalg.norm(x, axis=1))
    assert abs(rel8 - 0.0849) < 0.005, rel8
    assert abs(rel7 - 0.0954) < 0.005, rel7


# --------------------------------------------------------------------------- Q8 quantizers
def test_q8_0_roundtrip_bound(orc):
    """[minfer] s1: the error is bounded by half a scale step per value.  With the f32
    d = amax/127 that holds as stated; with the stored f16 d the bound grows by
    127*|d - f16(d)| (the step itself is rounded)."""
    x = workloads.activations_f32(16, 4096, seed=5)
    q = orc.quantize("q8_0", x)
    codes = orc.codes("q8_0", q, 4096).reshape(-1, 32).astype(np.float64)
    xb = x.reshape(-1, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=1)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    dh = d32.astype(np.float16).astype(np.float64)
    slack = 4e-7 * np.abs(xb)
    assert np.all(np.abs(xb - d32[:, None] * codes) <= d32[:, None] / 2 + slack)
    vals = orc.dequantize("q8_0", q, 4096).reshape(-1, 32)
    assert np.all(np.abs(xb - vals) <= d32[:, None] / 2 + 127 * np.abs(d32 - dh)[:, None] + slack)
    # the extreme lands on +-127, and the quantizer is odd-symmetric
    r = np.arange(xb.shape[0])
    assert np.all(np.abs(codes[r, np.abs(xb).argmax(axis=1)]) == 127)
    qn = orc.codes("q8_0", orc.quantize("q8_0", -x), 4096).reshape(-1, 32)
    assert np.array_equal(qn, -codes)


def test_q8_ties_to_even(orc):
    """[minfer] s3.2 (quantize_avx2): the code is x*id rounded to nearest with ties to even.
    A block whose amax is 127 has id = 1, so its half-integer inputs are exact ties."""
    rows = read_golden("q8_ties_to_even.txt")
    for t, bs in (("q8_0", 32), ("q8_K", 256)):
        x = np.zeros(bs, dtype=np.float32)
        for i, (v, _) in enumerate(rows):
            x[i] = float(v)
        c = orc.codes(t, orc.quantize(t, x), bs)[0]
        for i, (_, want) in enumerate(rows):
            assert c[i] == int(want), (t, i, c[i], want)


def test_zero_block_guard(orc):
    """[minfer] s3.2: an all-zero block gives d = 0 and codes 0, never NaN."""
    x = np.zeros((2, 512), dtype=np.float32)
    x[1, 256:] = 1.0                       # second row: one zero super-block, one not
    for t in ("q8_0", "q8_K"):
        q = orc.quantize(t, x)
        v = orc.dequantize(t, q, 512)
        assert np.all(np.isfinite(v))
        assert np.all(v[0] == 0) and np.all(v[1, :256] == 0)
        assert np.all(orc.codes(t, q, 512)[0] == 0)
    q = orc.quantize("q8_0", x[:1])
    assert np.all(q[0, ::34] == 0) and np.all(q[0, 1::34] == 0)
    w = orc.quantize("q4_0", workloads.weights_f32(3, 512, seed=1))
    y = orc.matmul("q4_0", w, q, 1, 3, 512)
    assert np.all(y == 0.0)


def test_q8_K_bsums_and_scale(orc):
    """[minfer] s3.2 (quantize_row_q8_k_buf): bsums[g] is the exact sum of the 16 saturated
    codes of group g; d is an f32 with 127*d = amax up to one rounding; error <= d/2.
    (With id = 127/amax, |x*id| never rounds past 127, so the saturation never fires.)"""
    x = workloads.activations_f32(8, 4096, seed=9)
    q = orc.quantize("q8_K", x)
    blocks = q.reshape(-1, 292)
    codes = blocks[:, 4:260].view(np.int8).astype(np.int64)
    bsums = blocks[:, 260:292].copy().view(np.int16).astype(np.int64)
    assert np.array_equal(bsums, codes.reshape(-1, 16, 16).sum(axis=2))
    d = blocks[:, 0:4].copy().view(np.float32).reshape(-1).astype(np.float64)
    amax = np.abs(x.reshape(-1, 256)).max(axis=1).astype(np.float64)
    assert np.all(np.abs(d * 127 - amax) <= 2 * np.spacing(amax.astype(np.float32)).astype(np.float64))
    xb = x.reshape(-1, 256).astype(np.float64)
    assert np.all(np.abs(xb - d[:, None] * codes) <= d[:, None] / 2 + 4e-7 * np.abs(xb))
    assert codes.max() <= 127 and codes.min() >= -127


def test_integer_inputs_are_exact(orc):
    """Textbook special case: integer inputs with a +-127 in every block give d = 1 exactly
    and codes equal to the inputs; the Q8_0 x Q8_0 product is then the integer matmul, which
    numpy computes exactly in int64 (all partial sums stay below 2^24)."""
    g = np.random.default_rng(4)
    M, N, K = 3, 5, 256
    w = g.integers(-127, 128, size=(N, K)).astype(np.float32)
    x = g.integers(-127, 128, size=(M, K)).astype(np.float32)
    w.reshape(N, -1, 32)[:, :, 0] = 127
    x.reshape(M, -1, 32)[:, :, 3] = -127
    wq = orc.quantize("q8_0", w)
    xq = orc.quantize("q8_0", x)
    assert np.array_equal(orc.codes("q8_0", wq, K), w.astype(np.int32))
    assert np.all(wq.reshape(-1, 34)[:, 0] == 0x00) and np.all(wq.reshape(-1, 34)[:, 1] == 0x3C)
    y = orc.matmul("q8_0", wq, xq, M, N, K)
    want = x.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(y.astype(np.int64), want)
    # the same for Q8_K activations with every super-block's scale exactly 1
    x2 = g.integers(-127, 128, size=(2, 512)).astype(np.float32)
    x2.reshape(2, -1, 256)[:, :, 7] = 127
    q2 = orc.quantize("q8_K", x2).reshape(-1, 292)
    assert np.all(q2[:, 0:4].copy().view(np.float32) == 1.0)
    assert np.array_equal(q2[:, 4:260].view(np.int8).reshape(2, 512), x2.astype(np.int8))


# --------------------------------------------------------------------------- K-quant decode
def test_q2_K_handmade_block(orc):
    """[ggml] s1.2: Q2_K decodes as d*sc*q - dmin*m with sc/m the low/high nibble of
    scales[g]; byte layout scales@0, qs@16, d@80, dmin@82 (84 B)."""
    blk = np.zeros(84, dtype=np.uint8)
    elems = []
    for row in read_golden("q2_K_handmade.txt"):
        if row[0] == "d_bits":
            v = int(row[1], 16); blk[80], blk[81] = v & 0xFF, v >> 8
        elif row[0] == "dmin_bits":
            v = int(row[1], 16); blk[82], blk[83] = v & 0xFF, v >> 8
        elif row[0] == "scale":
            blk[int(row[1])] = int(row[2], 16)
        elif row[0] == "qbyte":
            blk[16 + int(row[1])] = int(row[2], 16)
        elif row[0] == "elem":
            elems.append((int(row[1]), int(row[2]), float(row[4])))
    vals = orc.dequantize("q2_K", blk, 256)[0]
    codes = orc.codes("q2_K", blk, 256)[0]
    for e, c, want in elems:
        assert codes[e] == c and vals[e] == want, (e, codes[e], vals[e], want)


def test_q4_K_handmade_block(orc):
    """[minfer] s3.2 (the K-quant dot walked): value = q*d*sc_s - dmin*m_s; low nibbles of
    chunk j pair with elements 64j+l, high nibbles with 64j+32+l."""
    blk = np.zeros(144, dtype=np.uint8)
    elems = []
    for row in read_golden("q4_K_handmade.txt"):
        if row[0] == "d_bits":
            v = int(row[1], 16); blk[0], blk[1] = v & 0xFF, v >> 8
        elif row[0] == "dmin_bits":
            v = int(row[1], 16); blk[2], blk[3] = v & 0xFF, v >> 8
        elif row[0] == "sbyte":
            blk[4 + int(row[1])] = int(row[2])
        elif row[0] == "qbyte":
            blk[16 + int(row[1])] = int(row[2], 16)
        elif row[0] == "elem":
            elems.append((int(row[1]), int(row[2]), float(row[4])))
    vals = orc.dequantize("q4_K", blk, 256)[0]
    codes = orc.codes("q4_K", blk, 256)[0]
    for e, c, want in elems:
        assert codes[e] == c and vals[e] == want, (e, codes[e], vals[e], want)


def test_q5_q4_1_handmade_blocks(orc):
    """Hand-built Q5_0, Q5_1, Q4_1 and Q5_K blocks decode to the values worked out by hand:
    the fifth-bit plane, the nibble pairing and the min of each layout (GGUF readings; sizes
    [minfer] s1, s3.2)."""
    blocks = []
    for row in read_golden("q5_q4_1_handmade.txt"):
        if row[0] == "blk":
            blocks.append((row[1], np.zeros(int(row[2]), dtype=np.uint8), []))
        elif row[0] == "byte":
            blocks[-1][1][int(row[1])] = int(row[2], 0)
        elif row[0] == "elem":
            blocks[-1][2].append((int(row[1]), int(row[2]), float(row[3])))
    assert [b[0] for b in blocks] == ["q5_0", "q5_1", "q4_1", "q5_K"]
    for t, blk, elems in blocks:
        bv = orc.block_values(t)
        vals = orc.dequantize(t, blk, bv)[0]
        codes = orc.codes(t, blk, bv)[0]
        for e, code, want in elems:
            stored = codes[e] + 16 if t == "q5_0" else codes[e]
            assert stored == code and vals[e] == want, (t, e, stored, code, vals[e], want)


def test_q5_q4_1_integer_grids_are_exact(orc):
    """Textbook special case of the 32-value quantizers (readings): a block that is already an
    integer grid comes back exactly.  Q4_1 on c + {0..15} and Q5_1 on c + {0..31} have d = 1,
    m = c; Q5_0 on {-16..15} has its extreme -16 at code 0 and d = 1.  Each block is a
    permutation, so a misplaced nibble or high bit changes a value."""
    g = np.random.default_rng(8)
    for t, levels, c in (("q4_1", 16, 3.0), ("q5_1", 32, -5.0), ("q5_0", 32, -16.0)):
        base = np.arange(32) % levels
        x = np.stack([g.permutation(base) for _ in range(6)]).astype(np.float32) + np.float32(c)
        v = orc.dequantize(t, orc.quantize(t, x), 32)
        assert np.array_equal(v.reshape(x.shape), x.astype(np.float64)), t


@pytest.mark.parametrize("wtype", ["q4_1", "q5_0", "q5_1"])
def test_32_value_roundtrip(orc, wtype):
    """The 32-value quantizers (readings): every code in range; min/max grids reconstruct each
    value within half a step plus the f16 rounding of d and m; Q5_0's extreme sits at code -16
    (the Q4_0 idea, [ggml] s1.1) and the rest within half a step except the clipped end."""
    w = workloads.weights_f32(16, 512, seed=23, row_jitter=True)
    q = orc.quantize(wtype, w)
    v = orc.dequantize(wtype, q, 512).reshape(-1, 32)
    codes = orc.codes(wtype, q, 512).reshape(-1, 32)
    wb = w.reshape(-1, 32).astype(np.float64)
    lo, hi = {"q4_1": (0, 15), "q5_0": (-16, 15), "q5_1": (0, 31)}[wtype]
    assert codes.min() >= lo and codes.max() <= hi
    if wtype == "q5_0":
        r = np.arange(wb.shape[0])
        imax = np.abs(wb).argmax(axis=1)
        assert np.all(codes[r, imax] == -16)
        d32 = wb[r, imax] / -16
        dh = q.reshape(-1, 22)[:, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
        t = wb / d32[:, None]                  # the code each value wants, before clipping
        ok = t < 15.5
        bound = 0.5 * np.abs(dh)[:, None] + np.abs(t) * np.abs(dh - d32)[:, None] + 1e-6 * np.abs(wb)
        assert np.all((np.abs(v - wb) <= bound)[ok])
    else:
        step = (wb.max(axis=1) - wb.min(axis=1)) / (hi - lo)
        bound = 0.5 * step * (1 + 2e-3) + 2 ** -11 * np.abs(wb.min(axis=1)) + 1e-7
        assert np.all(np.abs(v - wb) <= bound[:, None]), np.abs(v - wb).max()


def test_q4_K_scale_packing_roundtrip(orc):
    """The 12-byte packing (reading: GGUF) is a bijection on eight 6-bit scales and mins:
    every value 0..63 in every slot survives pack (via the quantizer) and unpack.  Checked by
    crafting sub-blocks whose quantized scales and mins take chosen values."""
    g = np.random.default_rng(12)
    for _ in range(20):
        blk = g.integers(0, 256, size=12, dtype=np.uint8)
        sc, mn = orc.q4_K_scales(blk.tobytes())
        assert sc.min() >= 0 and sc.max() <= 63 and mn.min() >= 0 and mn.max() <= 63
    # the unpack reaches every (slot, value): the low sub-blocks read 6 plain bits
    seen = set()
    for s in range(8):
        for v in range(64):
            b = np.zeros(12, dtype=np.uint8)
            if s < 4:
                b[s] = v
            else:
                b[s + 4] = v & 15
                b[s - 4] = (v >> 4) << 6
            sc, _ = orc.q4_K_scales(b.tobytes())
            assert sc[s] == v and np.count_nonzero(sc) == (v != 0)
            seen.add((s, v))
    assert len(seen) == 512


@pytest.mark.parametrize("wtype", ["q4_K", "q2_K", "q6_K", "q5_K"])
def test_kquant_roundtrip(orc, wtype):
    """K-quant weight quantizers (readings): codes in range and every value reconstructed
    within the grid's step plus the rounding of its stored scale and min.  A wrong pack or
    unpack (swapped nibbles, shifted codes, wrong group) breaks this by a wide margin."""
    w = workloads.weights_f32(16, 1024, seed=21, row_jitter=True)
    q = orc.quantize(wtype, w)
    v = orc.dequantize(wtype, q, 1024)
    codes = orc.codes(wtype, q, 1024)
    lo, hi = {"q4_K": (0, 15), "q2_K": (0, 3), "q6_K": (-32, 31), "q5_K": (0, 31)}[wtype]
    assert codes.min() >= lo and codes.max() <= hi
    err = np.abs(v - w)
    gsz = 32 if wtype in ("q4_K", "q5_K") else 16
    rng_ = w.reshape(-1, gsz).max(axis=1) - np.minimum(w.reshape(-1, gsz).min(axis=1), 0)
    levels = {"q4_K": 15, "q2_K": 3, "q6_K": 63, "q5_K": 31}[wtype]
    step = rng_ / levels
    # a step and a half covers the grid offset from the rounded 6/4-bit scale and min
    assert np.all(err.reshape(-1, gsz) <= 1.5 * step[:, None] + 1e-6), err.max()
    rel = np.linalg.norm(v - w) / np.linalg.norm(w)
    assert rel < {"q4_K": 0.12, "q2_K": 0.45, "q6_K": 0.03, "q5_K": 0.06}[wtype], rel


def test_q6_K_extreme_code(orc):
    """Q6_K quantizer (reading, the Q4_0 idea on 6 bits): the signed extreme of each group of
    16 maps to the stored code 0 (value -32 * d * sc)."""
    w = workloads.weights_f32(4, 512, seed=3)
    q = orc.quantize("q6_K", w)
    codes = orc.codes("q6_K", q, 512).reshape(-1, 16)
    wb = w.reshape(-1, 16)
    imax = np.abs(wb).argmax(axis=1)
    assert np.all(codes[np.arange(codes.shape[0]), imax] == -32)


# --------------------------------------------------------------------------- dots
def _inputs(wtype, M, N, K, seed, orc):
    w = workloads.weights_f32(N, K, seed, row_jitter=True)
    x = workloads.activations_f32(M, K, seed)
    return orc.quantize(wtype, w), orc.quantize(orc.act_type(wtype), x)


@pytest.mark.parametrize("wtype", QTYPES)
def test_factorized_equals_bruteforce(orc, wtype):
    """[ggml] s2: multiplying codes as integers and applying the two scales once per block
    is exact.  So the factorized sum in binary64 equals the brute-force dequantized dot to
    double rounding, and the pages' fp32 fold is within fp32 accumulation error of it.  The
    brute force decodes every element on its own path, so a wrong nibble pairing, a dropped
    min term, a sign slip or a transposed operand in the kernel arithmetic fails here."""
    bv = 256 if wtype in KQUANTS else 32
    for K in sorted({bv, 2 * bv, 512 if bv == 32 else 768}):
        for N in (1, 3, 7):
            M = 3
            W, X = _inputs(wtype, M, N, K, 100 + K + N, orc)
            yb = orc.matmul_exact(wtype, W, X, M, N, K, bruteforce=True)
            ye = orc.matmul_exact(wtype, W, X, M, N, K)
            y = orc.matmul(wtype, W, X, M, N, K)
            wv = orc.dequantize(wtype, W, K)
            xv = orc.dequantize(orc.act_type(wtype), X, K)
            mag = np.abs(xv) @ np.abs(wv).T          # sum of |terms|
            assert np.all(np.abs(ye - yb) <= 1e-13 * mag + 1e-300)
            assert np.all(np.abs(y - yb) <= 2e-6 * mag + 1e-30)
            # and against a float64 BLAS product of the dequantized operands
            assert np.allclose(xv @ wv.T, yb, rtol=0, atol=1e-12 * mag.max())


@pytest.mark.parametrize("wtype", QTYPES)
def test_blocksums_consistent(orc, wtype):
    """The integer block sums reassemble the exact dot: sum_b dw*dx*isum_b (32-value types) and
    the two-term K-quant fold (value, min) equal the brute force; Q6_K's value - 32*min is the
    signed-code sum ([minfer] s3.2: Sum((q*d_s - m_s)*a) = d_s*Sum(q*a) - m_s*Sum(a))."""
    K = 512
    M, N = 2, 3
    W, X = _inputs(wtype, M, N, K, 55, orc)
    s = orc.blocksums(wtype, W, X, M, N, K).astype(np.float64)
    yb = orc.matmul_exact(wtype, W, X, M, N, K, bruteforce=True)
    wb = W.reshape(N, -1, orc.block_bytes(wtype))
    xb = X.reshape(M, -1, orc.block_bytes(orc.act_type(wtype)))
    h = lambda a: a.copy().view(np.float16).astype(np.float64)[..., 0]
    if wtype not in KQUANTS:
        dw, dx = h(wb[:, :, 0:2]), h(xb[:, :, 0:2])
        y = np.einsum("tob,ob,tb->to", s, dw, dx)
        if wtype in ("q4_1", "q5_1"):   # the min meets the activation block's code sum
            asum = xb[:, :, 2:34].view(np.int8).astype(np.float64).sum(axis=2)
            y += np.einsum("tb,ob,tb->to", asum, h(wb[:, :, 2:4]), dx)
    else:
        dx = xb[:, :, 0:4].copy().view(np.float32).astype(np.float64)[..., 0]
        off = {"q4_K": (0, 2), "q2_K": (80, 82), "q6_K": (208, None), "q5_K": (0, 2)}[wtype]
        dw = h(wb[:, :, off[0]:off[0] + 2])
        v, m = s[:, :, 0::2], s[:, :, 1::2]
        if wtype == "q6_K":
            y = np.einsum("tob,ob,tb->to", v - 32 * m, dw, dx)
        else:
            dmin = h(wb[:, :, off[1]:off[1] + 2])
            y = np.einsum("tob,ob,tb->to", v, dw, dx) - np.einsum("tob,ob,tb->to", m, dmin, dx)
    assert np.allclose(y, yb, rtol=1e-12, atol=1e-15)


def test_thread_invariance(orc):
    """[minfer] s3.2 thread pool / [krafla] Threads: each output row belongs to one worker,
    so the result is bit-identical for any thread count."""
    for wtype in QTYPES:
        K = 512
        W, X = _inputs(wtype, 2, 37, K, 77, orc)
        ys = [orc.matmul(wtype, W, X, 2, 37, K, nthreads=n) for n in (1, 2, 5, 8)]
        for y in ys[1:]:
            assert np.array_equal(y.view(np.uint32), ys[0].view(np.uint32))


def test_token_major_output(orc):
    """[minfer] s3.4 (the transposed-output bug): out is [nt][od]; with nt > 1 row t of the
    output must be the matvec of token t alone."""
    K, N, M = 256, 9, 4
    W, X = _inputs("q4_0", M, N, K, 8, orc)
    y = orc.matmul("q4_0", W, X, M, N, K)
    for t in range(M):
        yt = orc.matmul("q4_0", W, X[t:t + 1], 1, N, K)
        assert np.array_equal(y[t], yt[0])


def test_get_rows_returns_the_rows_asked_for(orc):
    """[minfer] s3.2, "The embedding 'matmul'": token id r reads row r.  Rows of integers with
    |max| = 127 quantize to Q8_0 with d = 1 exactly, so each looked-up row is its source row, in
    the order the ids give, repeats included."""
    N, K = 9, 64
    rng = np.random.default_rng(5)
    w = rng.integers(-126, 127, size=(N, K)).astype(np.float32)
    w[:, 0] = w[:, 32] = 127.0    # one 127 in each 32-value block
    w[np.arange(N), 1 + np.arange(N)] = -100.0 - np.arange(N)   # every row distinct
    W = orc.quantize("q8_0", w)
    ids = [4, 0, 8, 4, 2]
    assert np.array_equal(orc.get_rows("q8_0", W, ids, K), w[ids].astype(np.float64))
    with pytest.raises(IndexError):
        orc.get_rows("q8_0", W, [N], K)


# --------------------------------------------------------------------------- Q8 KV cache
def test_kv_row_size(orc):
    """[krafla] "Architecture", Attention: 68 bytes per head at head_dim 64 against 256 in f32,
    about 3.8x smaller."""
    for _, hd, b8, b32, shrink in read_golden("kv_cache.txt"):
        assert orc.kv_row_bytes(int(hd)) == int(b8)
        assert 4 * int(hd) == int(b32) and round(int(b32) / int(b8), 1) == float(shrink)


def test_kv_quantize_is_the_activation_rule(orc):
    """[krafla] "Architecture", Attention: K, V and the query heads use the activations'
    quantization rule.  Over 256 values that rule, with its f32 scale, is Q8_K's: codes and d
    equal Q8_K's bytes; over 32 values the codes equal Q8_0's and Q8_0's f16 scale is the
    f16 rounding of the f32 d."""
    x = workloads.activations_f32(6, 256, seed=41)
    x[0] = 0.0
    kv = orc.kv_quantize(x, 256)
    q8k = orc.quantize("q8_K", x).reshape(6, 292)
    assert np.array_equal(kv[:, 0:4], q8k[:, 0:4]) and np.array_equal(kv[:, 4:], q8k[:, 4:260])
    x32 = x[:, :32]
    kv32 = orc.kv_quantize(x32, 32)
    q80 = orc.quantize("q8_0", x32).reshape(6, 34)
    assert np.array_equal(kv32[:, 4:], q80[:, 2:])
    d = kv32[:, 0:4].copy().view(np.float32)[:, 0]
    assert np.array_equal(d.astype(np.float16).view(np.uint16), q80[:, 0:2].copy().view(np.uint16)[:, 0])


def _kv_integer_case(g, rows, hd):
    """Integer head vectors with |max| = 127 in each: scale exactly 1, codes = the integers."""
    v = g.integers(-127, 128, size=(rows, hd)).astype(np.float32)
    v[:, 0] = 127.0
    return v


def test_kv_scores_integer_case_and_head_mapping(orc):
    """Integer head vectors with scale 1: each score is the exact integer dot (numpy int64) times
    the power-of-two factor.  Query head h reads KV head h // (Hq // Hkv) ([krafla] "Architecture",
    "Data flow for one token"): with KV head 1's codes zeroed except the forced 127, query heads 2
    and 3 score only that element."""
    g = np.random.default_rng(42)
    Hq, Hkv, P, hd = 4, 2, 5, 64
    q = _kv_integer_case(g, Hq, hd)
    k = _kv_integer_case(g, P * Hkv, hd)
    k.reshape(P, Hkv, hd)[:, 1, 1:] = 0.0
    q8, k8 = orc.kv_quantize(q, hd), orc.kv_quantize(k, hd)
    s = orc.kv_scores(q8, k8, Hq, Hkv, P, hd, scale=0.125)
    kk = k.reshape(P, Hkv, hd).astype(np.int64)
    for h in range(Hq):
        want = kk[:, h // 2, :] @ q[h].astype(np.int64)
        assert np.array_equal(s[h].astype(np.float64), want * 0.125), h
    assert np.array_equal(s[2:].astype(np.float64), 127.0 * 127.0 * 0.125 * np.ones((2, P)))


def test_kv_wsum_matches_dequantized_einsum(orc):
    """The V sum equals a float64 einsum of the softmax-like weights and the dequantized V rows
    (a library product), with heads mapped as for the scores."""
    g = np.random.default_rng(43)
    Hq, Hkv, P, hd = 8, 2, 37, 32
    v = g.standard_normal((P * Hkv, hd)).astype(np.float32)
    v8 = orc.kv_quantize(v, hd)
    w = g.random((Hq, P)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    got = orc.kv_wsum(w, v8, Hq, Hkv, P, hd)
    dv = v8[:, 0:4].copy().view(np.float32)[:, 0].astype(np.float64)
    vq = v8[:, 4:].view(np.int8).astype(np.float64) * dv[:, None]
    vq = vq.reshape(P, Hkv, hd)
    want = np.stack([w[h].astype(np.float64) @ vq[:, h // (Hq // Hkv), :] for h in range(Hq)])
    assert np.allclose(got, want, rtol=1e-13, atol=1e-15)
    # the dequantized rows are within half a step of the f32 inputs
    assert np.all(np.abs(vq.reshape(-1, hd) - v) <= dv[:, None] / 2 * (1 + 1e-6) + 1e-12)


# --------------------------------------------------------------------------- RMSNorm
def test_rmsnorm_matches_float64(orc):
    """h = rmsnorm(x) ahead of the quantizer ([krafla] "Architecture", "Data flow for one token"),
    reading x * w / sqrt(mean(x^2) + eps): the f32 result is within 6e-7 of a float64 evaluation
    per element (8 single roundings of 2^-24 after a binary64 sum of squares that is exact to far
    below that), for an eps that matters and one that does not."""
    g = np.random.default_rng(60)
    for K, eps in ((4096, 1e-6), (896, 0.5), (256, 1e-5)):
        x = workloads.activations_f32(3, K, seed=K)
        w = g.uniform(0.25, 2.0, size=K).astype(np.float32)
        h = orc.rmsnorm(x, w, eps)
        x64 = x.astype(np.float64)
        ref = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + eps) * w
        assert np.all(np.abs(h - ref) <= 6e-7 * np.abs(ref) + 1e-30), np.max(np.abs(h - ref) / np.abs(ref))


def test_rmsnorm_exact_cases(orc):
    """A constant power-of-two vector with eps = 0 normalizes to -w exactly, and scaling x by a
    power of two leaves h unchanged bit for bit (every step scales exactly)."""
    K = 512
    w = np.random.default_rng(61).uniform(0.5, 1.5, size=K).astype(np.float32)
    x = np.full((1, K), -0.5, dtype=np.float32)
    assert np.array_equal(orc.rmsnorm(x, w, 0.0)[0], -w)
    y = workloads.activations_f32(2, K, seed=62)
    assert np.array_equal(orc.rmsnorm(y, w, 0.0).view(np.uint32), orc.rmsnorm(y * 4, w, 0.0).view(np.uint32))
