"""Integer-exact parity of every production multiply path against the oracle, for all nine weight
formats.

[krafla] "Architecture", Numerics (integer matvec: the block sums are exact) and [minfer] s3.2 (the
scalar kernel: the i32 accumulator never rounds) make each block's integer dot product exact; the
pages' fold then scales it once per block.  Here the block bytes are hand-made: random code bytes
and sub-block scale bytes, with every f16 scale field (d, and dmin or m where the format has one)
set to 0 or +-1/2 or +-1, and every activation scale to 1/2 or 1.  Each block's contribution is then
an exact multiple of 1/4, and the inputs are sized so that the sum of the magnitudes of all
contributions to one output stays below 2^22: every partial sum, in any order, is exact in f32.  So
y is one exact number and the GPU must reproduce the oracle's y bit for bit, through the decoders
the production kernels use (the super-unit decoders at K % 256 == 0, the per-block ones otherwise,
the segmented rows at K = 12288, the fused quantizer, the grouped launch and both tensor-core
prefills).  A decoder slip -- a wrong code, nibble, bit plane, scale, min or sign -- changes an
integer and shows up as a different y."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu

WTYPES = ["q4_0", "q8_0", "q4_1", "q5_0", "q5_1", "q4_K", "q5_K", "q6_K", "q2_K"]

# block values, block bytes, byte offsets of the f16 scale fields (the layouts of include/qmm.h)
FIELDS = {"q4_0": (32, 18, (0,)), "q8_0": (32, 34, (0,)), "q4_1": (32, 20, (0, 2)), "q5_0": (32, 22, (0,)),
          "q5_1": (32, 24, (0, 2)), "q4_K": (256, 144, (0, 2)), "q5_K": (256, 176, (0, 2)),
          "q6_K": (256, 210, (208,)), "q2_K": (256, 84, (80, 82))}
# the largest integer one weight value contributes per unit of |a| (value part plus min part):
# Q4_0 |q-8|, Q8_0 |q|, Q4_1 q + 1 (the min scales sum(a)), Q5_0 |q-16|, Q5_1 q + 1,
# Q4_K sc*q + m = 63*15 + 63, Q5_K 63*31 + 63, Q6_K |sc|*63 + 32*|sc| (stored codes and the -32
# through the bsums), Q2_K 15*3 + 15
def w_int_max(wtype, q6_scale):
    return {"q4_0": 8, "q8_0": 128, "q4_1": 16, "q5_0": 16, "q5_1": 32, "q4_K": 1008, "q5_K": 2016,
            "q6_K": 95 * q6_scale, "q2_K": 60}[wtype]


F16_SCALES = np.array([0x0000, 0x3800, 0x3C00, 0xB800, 0xBC00], dtype=np.uint16)  # 0, 1/2, 1, -1/2, -1
NNZ = 256  # small (+-1) activation codes per row


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    qmm.build()
    qmm.load()
    yield
    assert qmm.qmm_device_status(clear=True) == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def act_name(wtype):
    return "q8_0" if FIELDS[wtype][0] == 32 else "q8_K"


def hand_weights(wtype, N, K, seed, q6_scale=127):
    """N rows of random block bytes with power-of-two (or zero) f16 scale fields; Q6_K's int8
    sub-block scales drawn from [-q6_scale, q6_scale]."""
    g = np.random.default_rng(seed)
    bv, bb, f16s = FIELDS[wtype]
    nb = K // bv
    raw = g.integers(0, 256, size=(N, nb, bb), dtype=np.uint8)
    for off in f16s:
        bits = F16_SCALES[g.integers(0, len(F16_SCALES), size=(N, nb))]
        raw[:, :, off:off + 2] = bits.view(np.uint8).reshape(N, nb, 2)
    if wtype == "q6_K":
        raw[:, :, 192:208] = g.integers(-q6_scale, q6_scale + 1, size=(N, nb, 16)).astype(np.int8).view(np.uint8)
    return raw.reshape(N, nb * bb)


def sparse_codes(M, K, g):
    """int codes: NNZ entries of +-1 per row at random positions, zeros elsewhere."""
    a = np.zeros((M, K), dtype=np.int32)
    for t in range(M):
        pos = g.choice(K, size=min(NNZ, K), replace=False)
        a[t, pos] = g.choice([-1, 1], size=pos.size)
    return a


def hand_activations(act, M, K, seed):
    """Quantized activation rows built by hand: scale 1/2 or 1 per block, sparse +-1 codes, and for
    Q8_K the bsums of those codes."""
    g = np.random.default_rng(seed)
    a = sparse_codes(M, K, g)
    if act == "q8_0":
        nb = K // 32
        blk = np.zeros((M, nb, 34), dtype=np.uint8)
        blk[:, :, 0:2] = np.array([0x3800, 0x3C00], np.uint16)[g.integers(0, 2, size=(M, nb))].view(np.uint8).reshape(
            M, nb, 2)
        blk[:, :, 2:34] = a.reshape(M, nb, 32).astype(np.int8).view(np.uint8)
    else:
        nb = K // 256
        blk = np.zeros((M, nb, 292), dtype=np.uint8)
        blk[:, :, 0:4] = np.array([0.5, 1.0], np.float32)[g.integers(0, 2, size=(M, nb))].view(np.uint8).reshape(
            M, nb, 4)
        blk[:, :, 4:260] = a.reshape(M, nb, 256).astype(np.int8).view(np.uint8)
        bs = a.reshape(M, nb, 16, 16).sum(axis=3).astype(np.int16)
        blk[:, :, 260:292] = bs.view(np.uint8).reshape(M, nb, 32)
    return blk.reshape(M, -1), np.abs(a).sum(axis=1).max()


def integer_inputs_f32(act, M, K, seed):
    """f32 rows that the activation quantizer maps to d = 1 and codes equal to the values: a +-127
    in every block (the block maximum), sparse +-1 elsewhere."""
    g = np.random.default_rng(seed)
    a = sparse_codes(M, K, g)
    bv = 32 if act == "q8_0" else 256
    nb = K // bv
    where = g.integers(0, bv, size=(M, nb)) + np.arange(nb) * bv
    a[np.arange(M)[:, None], where] = g.choice([-127, 127], size=(M, nb))
    return a.astype(np.float32), np.abs(a).sum(axis=1).max()


def check_exact_budget(wtype, sum_abs_a, granularity, q6_scale=127):
    """Every partial sum is exact when all contributions are multiples of `granularity` and their
    magnitudes add up to less than 2^24 * granularity (the largest scale factor is 1)."""
    bound = w_int_max(wtype, q6_scale) * int(sum_abs_a)
    assert bound * 1.0 < 2.0 ** 24 * granularity, "inputs too large for an exact test: %d" % bound


def assert_exact(y_gpu, W, X, wtype, M, N, K):
    ref = oracle.matmul(wtype, W, X, M, N, K, nthreads=8)
    exact = oracle.matmul_exact(wtype, W, X, M, N, K)
    assert np.array_equal(ref.astype(np.float64), exact), "the oracle's own f32 fold is not exact here"
    got = np.asarray(y_gpu, dtype=np.float32).reshape(M, N)
    bad = got.view(np.uint32) != ref.view(np.uint32)
    assert not bad.any(), "%d outputs differ, first at %s: %r vs %r" % (
        bad.sum(), np.argwhere(bad)[0].tolist(), got[bad][:3], ref[bad][:3])


# ------------------------------------------------------------------ decode matvec on quantized rows
@pytest.mark.parametrize("wtype", WTYPES)
@pytest.mark.parametrize("N,K", [(1000, 4096), (77, 1024), (300, 12288), (131, 4064)])
def test_matvec_integer_exact(wtype, N, K):
    """qmm_matvec_<w>: K = 4096 / 1024 take the super-unit decoders of the 32-value formats, K = 4064
    (not a multiple of 256) their per-block decoders, K = 12288 rows cut into segments."""
    bv = FIELDS[wtype][0]
    if K % bv:
        pytest.skip("K is not a multiple of the block")
    W = hand_weights(wtype, N, K, seed=N + K)
    X, sa = hand_activations(act_name(wtype), 1, K, seed=K)
    check_exact_budget(wtype, sa, 0.25)
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    qmm.matvec(wtype, dev(W), dev(X), y, N, K)
    assert_exact(host(y), W, X, wtype, 1, N, K)


# ------------------------------------------------------------------ fused quantize + matvec, grouped
@pytest.mark.parametrize("wtype", WTYPES)
@pytest.mark.parametrize("M", [1, 3])
def test_linear_integer_exact(wtype, M):
    """qmm_linear_<w> from f32 rows: the in-kernel quantizer must produce d = 1 and the codes (the
    scratch rows are compared with the oracle's quantization too), then the exact y."""
    N, K = 515, 4096
    q6 = 24
    W = hand_weights(wtype, N, K, seed=11 + M, q6_scale=q6)
    x, sa = integer_inputs_f32(act_name(wtype), M, K, seed=12 + M)
    check_exact_budget(wtype, sa, 0.5, q6)
    X = oracle.quantize(act_name(wtype), x)
    sb = M * qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.linear(wtype, dev(W), dev(x), scratch, sb, y, M, N, K)
    assert np.array_equal(host(scratch), X.reshape(-1))
    assert_exact(host(y), W, X, wtype, M, N, K)


@pytest.mark.parametrize("wtype", WTYPES)
def test_linear_group_integer_exact(wtype):
    """qmm_linear_group: two matrices sharing one row in one launch per token."""
    K, Ns = 4096, (300, 77)
    q6 = 24
    x, sa = integer_inputs_f32(act_name(wtype), 1, K, seed=21)
    check_exact_budget(wtype, sa, 0.5, q6)
    X = oracle.quantize(act_name(wtype), x)
    Ws = [hand_weights(wtype, N, K, seed=22 + i, q6_scale=q6) for i, N in enumerate(Ns)]
    ys = [torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
    sb = qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    qmm.qmm_linear_group(wtype, [dev(W) for W in Ws], list(Ns), dev(x), scratch, sb, ys, 1, K)
    for W, y, N in zip(Ws, ys, Ns):
        assert_exact(host(y), W, X, wtype, 1, N, K)


# ------------------------------------------------------------------ prefill (tensor cores and fallback)
@pytest.mark.parametrize("wtype", WTYPES)
@pytest.mark.parametrize("M,N,K", [(130, 300, 4096), (8, 129, 2048), (5, 64, 2048)])
def test_matmul_integer_exact(wtype, M, N, K):
    """qmm_matmul_<w>: M >= 8 on the tensor cores (several tiles, a ragged last tile of rows and of
    tokens), M = 5 per-token matvecs."""
    W = hand_weights(wtype, N, K, seed=31 + M)
    X, sa = hand_activations(act_name(wtype), M, K, seed=32 + M)
    check_exact_budget(wtype, sa, 0.25)
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.matmul(wtype, dev(W), dev(X), Y, M, N, K)
    assert_exact(host(Y), W, X, wtype, M, N, K)


@pytest.mark.parametrize("wtype", WTYPES)
def test_linear_prefill_integer_exact(wtype):
    """qmm_linear_<w> with M >= 8: all rows quantized, then the tensor-core prefill."""
    M, N, K = 64, 200, 4096
    q6 = 24
    W = hand_weights(wtype, N, K, seed=41, q6_scale=q6)
    x, sa = integer_inputs_f32(act_name(wtype), M, K, seed=42)
    check_exact_budget(wtype, sa, 0.5, q6)
    X = oracle.quantize(act_name(wtype), x)
    sb = M * qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.linear(wtype, dev(W), dev(x), scratch, sb, Y, M, N, K)
    assert np.array_equal(host(scratch), X.reshape(-1))
    assert_exact(host(Y), W, X, wtype, M, N, K)


def test_hand_inputs_are_what_they_claim():
    """CPU-side check of the construction: the oracle reads the hand-made scale fields as the powers
    of two they were set to, and the activation quantizer maps the integer rows to d = 1."""
    W = hand_weights("q4_K", 3, 512, seed=1)
    d = W.reshape(3, 2, 144)[:, :, 0:2].copy().view(np.float16).astype(np.float64)
    assert set(np.unique(np.abs(d))) <= {0.0, 0.5, 1.0}
    x, _ = integer_inputs_f32("q8_0", 2, 256, seed=2)
    X = oracle.quantize("q8_0", x).reshape(2, 8, 34)
    assert np.all(X[:, :, 0:2].copy().view(np.float16) == 1.0)
    assert np.array_equal(X[:, :, 2:].view(np.int8).reshape(2, 256).astype(np.float32), x)
