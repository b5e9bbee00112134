"""The Q8 KV cache on the GPU against the CPU oracle ([krafla] "Architecture", Attention,
"Q8 cache"): quantized rows and scores bit-exact; the V sum within the a-priori bound of its
f32 summation, (P + 2) * 2^-24 * sum_p |w dv v| per output, and identical run to run."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu


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


def gpu_quantize(x, hd):
    rows = x.size // hd
    out = torch.empty(rows * qmm.qmm_kv_row_bytes(hd), dtype=torch.uint8, device="cuda")
    qmm.qmm_kv_quantize(dev(x.reshape(rows, hd)), out, rows, hd)
    return out


@pytest.mark.parametrize("rows,hd", [(1, 16), (7, 64), (40, 128), (33, 256), (9, 48)])
def test_kv_quantize_bitexact(rows, hd):
    x = workloads.activations_f32(rows, hd, seed=500 + hd)
    x[0] = 0.0                                   # all-zero vector: d = 0, codes 0
    if rows > 2:
        x[1] = 0.0
        x[1, 0], x[1, 1], x[1, 2] = 127.0, 2.5, -3.5   # exact ties at id = 1
    got = host(gpu_quantize(x, hd)).reshape(rows, -1)
    want = oracle.kv_quantize(x, hd)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5].tolist()


def test_kv_append_rows_at_4_byte_offsets():
    """Appending position p writes Hkv rows at byte p * Hkv * (4 + hd), 4-byte aligned only."""
    hd, Hkv, P = 64, 1, 5
    x = workloads.activations_f32(P * Hkv, hd, seed=77)
    rb = qmm.qmm_kv_row_bytes(hd)
    cache = torch.zeros(P * Hkv * rb, dtype=torch.uint8, device="cuda")
    for p in range(P):
        qmm.qmm_kv_quantize(dev(x[p * Hkv:(p + 1) * Hkv]), cache[p * Hkv * rb:], Hkv, hd)
    assert np.array_equal(host(cache).reshape(P * Hkv, rb), oracle.kv_quantize(x, hd))


SHAPES = [(32, 8, 4096, 128), (4, 4, 1, 64), (8, 1, 300, 64), (6, 3, 129, 16), (14, 2, 257, 256), (2, 2, 128, 32)]


@pytest.mark.parametrize("Hq,Hkv,P,hd", SHAPES)
def test_kv_scores_bitexact(Hq, Hkv, P, hd):
    q, k, _, _ = workloads.kv_inputs(Hq, Hkv, P, hd, seed=600 + P)
    q8, k8 = oracle.kv_quantize(q, hd), oracle.kv_quantize(k, hd)
    scale = float(np.float32(1.0 / np.sqrt(hd)))
    want = oracle.kv_scores(q8, k8, Hq, Hkv, P, hd, scale)
    s = torch.empty(Hq, P, dtype=torch.float32, device="cuda")
    qmm.qmm_kv_scores(dev(q8), dev(k8), s, Hq, Hkv, P, hd, scale)
    got = host(s)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), np.argwhere(got != want)[:5].tolist()


def _wsum_bound(w, v8, Hq, Hkv, P, hd):
    """(P + 2) * 2^-24 * sum_p |w dv v| per output: the a-priori bound of an f32 sum of P terms
    (each term a product rounded once) in any order."""
    dv = v8[:, 0:4].copy().view(np.float32)[:, 0].astype(np.float64)
    av = np.abs(v8[:, 4:].view(np.int8).astype(np.float64)) * np.abs(dv)[:, None]
    av = av.reshape(P, Hkv, hd)
    G = Hq // Hkv
    mag = np.stack([np.abs(w[h]).astype(np.float64) @ av[:, h // G, :] for h in range(Hq)])
    return (P + 2) * 2.0 ** -24 * mag


@pytest.mark.parametrize("Hq,Hkv,P,hd", SHAPES)
def test_kv_wsum_matches_oracle(Hq, Hkv, P, hd):
    _, _, v, w = workloads.kv_inputs(Hq, Hkv, P, hd, seed=700 + P)
    v8 = oracle.kv_quantize(v, hd)
    want = oracle.kv_wsum(w, v8, Hq, Hkv, P, hd)
    sb = qmm.qmm_kv_wsum_scratch_bytes(Hq, P, hd)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    out = torch.empty(Hq, hd, dtype=torch.float32, device="cuda")
    wd, vd = dev(w), dev(v8)
    qmm.qmm_kv_wsum(wd, vd, out, scratch, sb, Hq, Hkv, P, hd)
    got = host(out).astype(np.float64)
    bound = _wsum_bound(w, v8, Hq, Hkv, P, hd)
    assert np.all(np.abs(got - want) <= bound + 1e-30), np.max(np.abs(got - want) / (bound + 1e-30))
    # the typical error is far inside the bound: within 1e-5 of each head's output norm
    norm = np.linalg.norm(want, axis=1, keepdims=True)
    assert np.all(np.abs(got - want) <= 1e-5 * norm + 1e-30)
    out2 = torch.empty_like(out)
    qmm.qmm_kv_wsum(wd, vd, out2, scratch, sb, Hq, Hkv, P, hd)
    assert np.array_equal(host(out2).view(np.uint32), host(out).view(np.uint32))


def test_kv_gpu_quantized_cache_feeds_scores():
    """The whole path on the device: quantize q and K with qmm_kv_quantize, then score; equals the
    oracle on the same f32 inputs."""
    Hq, Hkv, P, hd = 16, 4, 200, 128
    q, k, _, _ = workloads.kv_inputs(Hq, Hkv, P, hd, seed=801)
    scale = float(np.float32(0.088))
    s = torch.empty(Hq, P, dtype=torch.float32, device="cuda")
    qmm.qmm_kv_scores(gpu_quantize(q, hd), gpu_quantize(k, hd), s, Hq, Hkv, P, hd, scale)
    want = oracle.kv_scores(oracle.kv_quantize(q, hd), oracle.kv_quantize(k, hd), Hq, Hkv, P, hd, scale)
    assert np.array_equal(host(s).view(np.uint32), want.view(np.uint32))
