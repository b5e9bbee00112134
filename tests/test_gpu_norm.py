"""RMSNorm fused ahead of the quantizer ([krafla] "Architecture", "Data flow for one token":
h = rmsnorm(x) ; qa = quantize_q8(h)) on the GPU against the CPU oracle.

The oracle sums the squares left to right in binary64 (the plain definition); the kernels sum them
in f32 in their own order, so the two scales s differ by a few units in the last place.  The codes
rne(h_i * 127/amax) do not depend on s beyond rounding (h and amax scale together), so they must be
bit-exact except where h_i * 127/amax lies within a few roundings of a tie, where +-1 is allowed and
counted; each block's d = amax/127 follows s and may differ by the derived bound.  The products are
within 1e-5 of each token row's L2 norm."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5


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
    return "q8_0" if wtype in ("q4_0", "q8_0", "q4_1", "q5_0", "q5_1") else "q8_K"


def assert_rows_close(y, ref, tol=TOL):
    y = np.asarray(y, dtype=np.float64).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    norm = np.linalg.norm(ref, axis=-1, keepdims=True)
    bad = np.abs(y - ref) > tol * norm + 1e-30
    assert not bad.any(), (np.abs(y - ref) / np.maximum(norm, 1e-30)).max()


# |t' - t| for t = h_i * 127/amax, |t| <= 127: h_i and amax each carry at most four roundings of
# 2^-24 relative on either side, id and the product one more each: about 11 * 2^-24 * 127 = 8.3e-5.
CODE_TIE_MARGIN = 2e-4


def scale_margin(K):
    """Relative bound on the difference of d = amax/127 between the two sums of squares: the kernel's
    f32 sum (sequential runs of 8, then a tree of depth log2(K/8)) is within (8 + log2 K) * 2^-24 of
    the exact sum, the oracle's within 2^-24; s = 1/sqrt(ss/K + eps) halves that and adds four
    roundings per side; amax and the division add three more.  Doubled for safety."""
    u = 2.0 ** -24
    return 2 * (0.5 * (9 + np.log2(K)) + 8 + 6) * u


def normed_codes_differences(act, got, h):
    """Compares the GPU's quantized normed rows `got` (bytes) with the oracle's quantization of the
    oracle's h.  Returns the number of codes that took the +-1 allowance near a tie."""
    M, K = h.shape
    bv, bb, off = (32, 34, 2) if act == "q8_0" else (256, 292, 4)
    want = oracle.quantize(act, h).reshape(M, K // bv, bb)
    got = np.asarray(got, dtype=np.uint8).reshape(M, K // bv, bb)
    cw = want[:, :, off:off + bv].view(np.int8).astype(np.int32)
    cg = got[:, :, off:off + bv].view(np.int8).astype(np.int32)
    hb = h.reshape(M, K // bv, bv).astype(np.float32)
    amax = np.abs(hb).max(axis=2, keepdims=True)
    with np.errstate(divide="ignore"):
        idv = np.where(amax > 0, np.float32(127.0) / amax, np.float32(0.0)).astype(np.float32)
    t = (hb * idv).astype(np.float32).astype(np.float64)
    near = np.abs(t - np.floor(t) - 0.5) <= CODE_TIE_MARGIN
    diff = cg - cw
    assert np.all(diff[~near] == 0), "codes differ away from a tie: %s" % np.argwhere((diff != 0) & ~near)[:5]
    assert np.all(np.abs(diff) <= 1)
    dm = scale_margin(K)
    a32 = amax[:, :, 0].astype(np.float64)
    if act == "q8_0":
        dwant = want[:, :, 0:2].copy().view(np.uint16)[:, :, 0].astype(np.int64)
        dgot = got[:, :, 0:2].copy().view(np.uint16)[:, :, 0].astype(np.int64)
        d32 = (amax[:, :, 0] / np.float32(127.0)).astype(np.float32).astype(np.float64)
        v = dwant.astype(np.uint16).view(np.float16).astype(np.float64)
        up = (dwant + 1).astype(np.uint16).view(np.float16).astype(np.float64)
        dn = np.maximum(dwant - 1, 0).astype(np.uint16).view(np.float16).astype(np.float64)
        near_d = (np.abs(d32 - (v + up) / 2) <= dm * d32) | (np.abs(d32 - (v + dn) / 2) <= dm * d32)
        dd = dgot - dwant
        assert np.all(dd[~near_d] == 0) and np.all(np.abs(dd) <= 1)
    else:
        dwant = want[:, :, 0:4].copy().view(np.float32)[:, :, 0].astype(np.float64)
        dgot = got[:, :, 0:4].copy().view(np.float32)[:, :, 0].astype(np.float64)
        assert np.all(np.abs(dgot - dwant) <= dm * dwant)
        bs_got = got[:, :, 260:292].copy().view(np.int16).astype(np.int32)
        assert np.array_equal(bs_got, cg.reshape(M, K // bv, 16, 16).sum(axis=3))  # bsums of its own codes
    assert np.all(cg[a32 == 0] == 0)  # an all-zero block stays all zero
    return int((diff != 0).sum())


def norm_weight(K, seed):
    return np.random.default_rng(seed).uniform(0.5, 1.5, size=K).astype(np.float32)


@pytest.mark.parametrize("act,M,K,eps", [("q8_0", 1, 4096, 1e-6), ("q8_0", 3, 896, 1e-5), ("q8_0", 2, 96, 0.5),
                                         ("q8_K", 5, 256, 1e-6), ("q8_K", 2, 12288, 1e-6), ("q8_0", 1, 65536, 1e-6),
                                         ("q8_K", 1, 65536, 0.0)])
def test_rmsnorm_quantize_bitexact(act, M, K, eps):
    x = workloads.activations_f32(M, K, seed=900 + K)
    if M >= 3:
        x[1] = 0.0 if eps > 0 else 1.0      # an all-zero row (eps keeps the scale finite)
        x[2] = -0.5                          # a constant row
    w = norm_weight(K, K)
    h = oracle.rmsnorm(x, w, eps)
    out = torch.empty(M * qmm.qmm_row_bytes(act, K), dtype=torch.uint8, device="cuda")
    qmm.qmm_rmsnorm_quantize(act, dev(x), dev(w), eps, out, M, K)
    flips = normed_codes_differences(act, host(out), h)
    print("%s M=%d K=%d: %d of %d codes took the +-1 allowance near a tie" % (act, M, K, flips, M * K))


@pytest.mark.parametrize("wtype,Ns,K,M", [("q8_0", (12288,), 4096, 1), ("q4_K", (300, 77, 1024), 4096, 1),
                                          ("q6_K", (257,), 12288, 2), ("q2_K", (129, 64), 1024, 1),
                                          ("q4_0", (64, 33), 896, 3), ("q5_1", (100,), 512, 1),
                                          ("q5_K", (333, 20), 4096, 2), ("q4_K", (512, 300), 4096, 16),
                                          ("q4_0", (512,), 4096, 16), ("q8_0", (300, 77), 2048, 16),
                                          ("q5_1", (130,), 1024, 9)])
def test_linear_norm_matches_oracle(wtype, Ns, K, M):
    """Decode tokens (one fused launch each) and the prefill route (M = 16: norm-quantize all rows,
    then the tensor-core matmul) against the oracle on the same f32 inputs; the scratch holds the
    quantized normed rows."""
    eps = 1e-6
    x = workloads.activations_f32(M, K, seed=950 + K)
    w = norm_weight(K, 7)
    h = oracle.rmsnorm(x, w, eps)
    X = oracle.quantize(act_name(wtype), h)
    Ws, refs = [], []
    for g, N in enumerate(Ns):
        Wq = oracle.quantize(wtype, workloads.weights_f32(N, K, seed=960 + g, row_jitter=True))
        Ws.append(dev(Wq))
        refs.append(oracle.matmul(wtype, Wq, X, M, N, K, nthreads=8))
    ys = [torch.empty(M, N, dtype=torch.float32, device="cuda") for N in Ns]
    sb = M * qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    qmm.qmm_linear_norm(wtype, Ws, Ns, dev(x), dev(w), eps, scratch, sb, ys, M, K)
    flips = normed_codes_differences(act_name(wtype), host(scratch), h)
    print("%s M=%d K=%d: %d codes took the +-1 allowance near a tie" % (wtype, M, K, flips))
    for g in range(len(Ns)):
        assert_rows_close(host(ys[g]), refs[g])


def test_linear_norm_equals_matvec_on_the_normed_row():
    """The fused launch gives, bit for bit, the plain matvec of the row it stored."""
    wtype, N, K = "q4_K", 4096, 4096
    x = workloads.activations_f32(1, K, seed=990)
    w = norm_weight(K, 8)
    Wd = dev(oracle.quantize(wtype, workloads.weights_f32(N, K, seed=991)))
    sb = qmm.qmm_row_bytes("q8_K", K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    y = torch.empty(1, N, dtype=torch.float32, device="cuda")
    qmm.qmm_linear_norm(wtype, [Wd], [N], dev(x), dev(w), 1e-6, scratch, sb, [y], 1, K)
    y2 = torch.empty(N, dtype=torch.float32, device="cuda")
    qmm.matvec(wtype, Wd, scratch, y2, N, K)
    assert np.array_equal(host(y).reshape(-1).view(np.uint32), host(y2).view(np.uint32))
