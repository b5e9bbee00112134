"""Every kernel family of the bounds-checked library build on small, odd shapes.

Run as its own process with QMM_LIBRARY naming the bounds-checked libqmm.so (built with
-DQMM_CHECK_BOUNDS, where every kernel checks the index ranges of its computed accesses and records
QMM_E_BOUNDS instead of touching memory outside a buffer): the results must match the CPU oracle as
in the normal tests, and the device status must stay QMM_OK, i.e. no check fired.  Used by
tests/test_gpu_checked_build.py; prints "checked build ok" on success."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402

import torch  # noqa: E402

import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

WTYPES = ["q4_0", "q8_0", "q4_1", "q5_0", "q5_1", "q4_K", "q5_K", "q6_K", "q2_K"]


def act_name(w):
    return "q8_0" if w in ("q4_0", "q8_0", "q4_1", "q5_0", "q5_1") else "q8_K"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def close(y, ref, tol=1e-5):
    ref = np.asarray(ref, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64).reshape(ref.shape)
    norm = np.linalg.norm(ref, axis=-1, keepdims=True)
    assert np.all(np.abs(y - ref) <= tol * norm + 1e-30), np.max(np.abs(y - ref) / np.maximum(norm, 1e-30))


def status(where):
    st = qmm.qmm_device_status(clear=True)
    assert st == 0, "device status %s after %s" % (qmm.STATUS.get(st, st), where)


def main():
    path = os.environ.get("QMM_LIBRARY", "")
    assert path.endswith(os.path.join("_build_checked", "libqmm.so")), path
    L = qmm.load()
    assert L._name == path
    torch.cuda.set_device(0)
    status("start")

    for t, M, K in (("q8_0", 3, 96), ("q8_0", 17, 544), ("q8_K", 3, 768)):
        x = workloads.activations_f32(M, K, seed=K)
        want = oracle.quantize(t, x)
        out = torch.empty(want.size, dtype=torch.uint8, device="cuda")
        qmm.quantize(t, dev(x), out, M, K)
        assert np.array_equal(host(out), want.reshape(-1)), t
    status("activation quantizers")

    for w in WTYPES:
        bv = 32 if act_name(w) == "q8_0" else 256
        for N, K in ((37, 2 * bv if bv == 256 else 96), (131, 2048), (5, 12288)):
            W = oracle.quantize(w, workloads.weights_f32(N, K, seed=N, row_jitter=True))
            Wg = torch.empty(W.size, dtype=torch.uint8, device="cuda")
            qmm.quantize(w, dev(workloads.weights_f32(N, K, seed=N, row_jitter=True)), Wg, N, K)
            assert np.array_equal(host(Wg), W.reshape(-1)), w
            for M in (1, 3):
                x = workloads.activations_f32(M, K, seed=N + K)
                X = oracle.quantize(act_name(w), x)
                ref = oracle.matmul(w, W, X, M, N, K, nthreads=8)
                if M == 1:
                    y = torch.empty(N, dtype=torch.float32, device="cuda")
                    qmm.matvec(w, dev(W), dev(X), y, N, K)
                    close(host(y), ref[0])
                sb = M * qmm.qmm_row_bytes(act_name(w), K)
                scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
                y = torch.empty(M, N, dtype=torch.float32, device="cuda")
                qmm.linear(w, dev(W), dev(x), scratch, sb, y, M, N, K)
                close(host(y), ref)
            bs_want = oracle.blocksums(w, W, oracle.quantize(act_name(w), workloads.activations_f32(2, K, 3)), 2, N, K)
            s = torch.empty(bs_want.size, dtype=torch.int32, device="cuda")
            qmm.qmm_blocksums(w, dev(W), dev(oracle.quantize(act_name(w), workloads.activations_f32(2, K, 3))), s, 2,
                              N, K)
            assert np.array_equal(host(s), bs_want.reshape(-1)), w
        status("matvec / linear / blocksums " + w)

        # the tensor-core prefill: several tiles and ragged edges
        M, N, K = 137, 257, 2048
        W = oracle.quantize(w, workloads.weights_f32(N, K, seed=5, row_jitter=True))
        X = oracle.quantize(act_name(w), workloads.activations_f32(M, K, seed=6))
        Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
        qmm.matmul(w, dev(W), dev(X), Y, M, N, K)
        close(host(Y), oracle.matmul(w, W, X, M, N, K, nthreads=8))
        status("prefill " + w)

        # grouped and normed linears
        K = 2048
        x = workloads.activations_f32(1, K, seed=7)
        g = np.random.default_rng(8).uniform(0.5, 1.5, size=K).astype(np.float32)
        Ns = (70, 33)
        Ws = [oracle.quantize(w, workloads.weights_f32(N, K, seed=9 + i)) for i, N in enumerate(Ns)]
        ys = [torch.empty(1, N, dtype=torch.float32, device="cuda") for N in Ns]
        sb = qmm.qmm_row_bytes(act_name(w), K)
        scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
        qmm.qmm_linear_group(w, [dev(a) for a in Ws], list(Ns), dev(x), scratch, sb, ys, 1, K)
        X = oracle.quantize(act_name(w), x)
        for Wq, y, N in zip(Ws, ys, Ns):
            close(host(y), oracle.matmul(w, Wq, X, 1, N, K))
        qmm.qmm_linear_norm(w, [dev(a) for a in Ws], list(Ns), dev(x), dev(g), 1e-6, scratch, sb, ys, 1, K)
        Xn = oracle.quantize(act_name(w), oracle.rmsnorm(x, g, 1e-6))
        for Wq, y, N in zip(Ws, ys, Ns):
            close(host(y), oracle.matmul(w, Wq, Xn, 1, N, K))
        status("grouped / normed linear " + w)

        # GetRows
        N, K = 11, 512
        W = oracle.quantize(w, workloads.weights_f32(N, K, seed=10))
        ids = np.array([3, 0, 10, 3, 7], dtype=np.int32)
        out = torch.empty(len(ids), K, dtype=torch.float32, device="cuda")
        qmm.qmm_get_rows(w, dev(W), dev(ids), out, len(ids), N, K)
        assert np.array_equal(host(out), oracle.get_rows(w, W, ids, K).astype(np.float32)), w
        status("get_rows " + w)

    # the Q8 KV cache at a ragged length
    Hq, Hkv, P, hd = 8, 2, 333, 64
    q, k, v, wts = workloads.kv_inputs(Hq, Hkv, P, hd, seed=11)
    rb = qmm.qmm_kv_row_bytes(hd)
    kc = torch.empty(P * Hkv * rb, dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    qmm.qmm_kv_quantize(dev(k), kc, P * Hkv, hd)
    qmm.qmm_kv_quantize(dev(v), vc, P * Hkv, hd)
    q8 = torch.empty(Hq * rb, dtype=torch.uint8, device="cuda")
    qmm.qmm_kv_quantize(dev(q), q8, Hq, hd)
    sc = torch.empty(Hq, P, dtype=torch.float32, device="cuda")
    qmm.qmm_kv_scores(q8, kc, sc, Hq, Hkv, P, hd, 0.125)
    assert np.array_equal(host(sc), oracle.kv_scores(host(q8), host(kc), Hq, Hkv, P, hd, 0.125))
    sbk = qmm.qmm_kv_wsum_scratch_bytes(Hq, P, hd)
    ks = torch.empty(sbk, dtype=torch.uint8, device="cuda")
    out = torch.empty(Hq, hd, dtype=torch.float32, device="cuda")
    qmm.qmm_kv_wsum(dev(wts), vc, out, ks, sbk, Hq, Hkv, P, hd)
    close(host(out), oracle.kv_wsum(wts, host(vc), Hq, Hkv, P, hd))
    status("kv cache")
    print("checked build ok")


if __name__ == "__main__":
    main()
