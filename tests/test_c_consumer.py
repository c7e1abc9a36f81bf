"""The C ABI used from plain C: tests/abi_consumer.c includes include/tg.h alone, is compiled
as strict C99 (gcc -pedantic -Werror) and linked against libtg.so, with no Python or PyTorch
on its path.  Its host planning outputs (page tables, split map, per-CTA plan) must equal the
oracle bit for bit; on a GPU its retained sets must equal the oracle's and its decode outputs
must meet the attention tolerance."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import synth
from oracle import tangram as otg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _consumer(lib, tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    so = lib.load()._name  # the loaded libtg.so
    exe = str(tmp_path_factory.mktemp("abi") / "abi_consumer")
    pkg = os.path.dirname(so)
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "abi_consumer.c"), "-o", exe,
           so, f"-Wl,-rpath,{pkg}", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


@pytest.fixture(scope="module")
def consumer(lib, tmp_path_factory):
    return _consumer(lib, tmp_path_factory)


def _write_inputs(d, w, N_CTA, Bhat, N):
    scale = 1.0 / math.sqrt(w.d)
    with open(os.path.join(d, "dims"), "w") as f:
        f.write(f"{w.batch} {w.H} {w.H_q} {w.H_p} {w.P} {w.d} {int(N.max())} {N_CTA} {w.alpha!r} "
                f"{int(w.cluster)} {scale!r}\n")
    np.asarray(Bhat[0], np.float32).tofile(os.path.join(d, "bhat.f32"))
    np.asarray(N, np.int32).tofile(os.path.join(d, "N.i32"))


def _read(d, name, dtype, shape=None):
    a = np.fromfile(os.path.join(d, name), dtype=dtype)
    return a if shape is None else a.reshape(shape)


def _check_host(d, w, N_CTA, Bhat, N):
    ref = otg.build_pages(1, w.batch, w.H, w.H_p, w.P, w.alpha, Bhat, N, w.cluster)
    assert np.array_equal(_read(d, "head_order.i32", np.int32), ref["order"][0])
    assert np.array_equal(_read(d, "ntok.i32", np.int32, (w.batch, w.H)), ref["ntok"][0])
    assert np.array_equal(_read(d, "Phi.i64", np.int64), ref["Phi"][0])
    assert np.array_equal(_read(d, "pt_off.i64", np.int64), ref["pt_off"])
    assert np.array_equal(_read(d, "pt_ids.i32", np.int32), ref["pt_ids"])
    S = _read(d, "S.i32", np.int32)
    assert S.tolist() == otg.split_map_row(ref["Phi"][0], N_CTA)
    want = otg.work_list(S, ref["ntok"][0], ref["order"][0], w.H_p)
    items = _read(d, "items.i32", np.int32).reshape(-1, 7)
    got = [[] for _ in range(N_CTA)]
    for c, b, h, t0, t1, part, nparts in items.tolist():
        got[c].append((b, h, t0, t1, nparts, part))
    assert got == [[(b, h, t0, t1, np_, p) for b, h, _j, _lst, t0, t1, np_, p in cta] for cta in want]
    return ref


@pytest.mark.parametrize("case", ["small", "small_clustered", "config1"])
def test_c_consumer_host_planning_matches_oracle(consumer, tmp_path, case):
    if case == "config1":
        w, N_CTA = synth.workload(1), 148
    else:
        w = synth.small(L=1, cluster=case == "small_clustered", alpha=1.5 if case == "small_clustered" else 1.0)
        N_CTA = 24
    Bhat, N = synth.budgets_hat(w), synth.contexts(w)
    _write_inputs(str(tmp_path), w, N_CTA, Bhat, N)
    r = subprocess.run([consumer, str(tmp_path)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    _check_host(str(tmp_path), w, N_CTA, Bhat, N)


def test_c_consumer_reports_a_refused_call(consumer, tmp_path):
    """A call the library refuses ends the program with the library's own message."""
    w = synth.small(L=1)
    Bhat, N = synth.budgets_hat(w), synth.contexts(w)
    _write_inputs(str(tmp_path), w, 1, Bhat, N)  # N_CTA < G: the split map is refused
    r = subprocess.run([consumer, str(tmp_path)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 1
    assert "tg_split_map" in r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["small", "config1"])
def test_c_consumer_compacts_and_decodes_on_the_gpu(consumer, tmp_path, case):
    import torch
    from gpu_helpers import OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS

    if case == "config1":
        w, N_CTA = synth.workload(1), 148
    else:
        w, N_CTA = synth.small(L=1, cluster=True, alpha=1.5), 24
    d = str(tmp_path)
    Bhat, N = synth.budgets_hat(w), synth.contexts(w)
    Nmax = int(N.max())
    _write_inputs(d, w, N_CTA, Bhat, N)
    s = synth.scores(w, 0, "cpu")[:, :, :Nmax].contiguous()
    K, V = synth.keys_values(w, 0, "cpu")
    K, V = K[:, :, :Nmax].contiguous(), V[:, :, :Nmax].contiguous()
    q = synth.queries(w, 0, "cpu")
    s.numpy().astype(np.float32).tofile(os.path.join(d, "scores.f32"))
    for name, t in (("K.u16", K), ("V.u16", V), ("q.u16", q)):
        t.view(torch.int16).numpy().tofile(os.path.join(d, name))
    r = subprocess.run([consumer, d, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    ref = _check_host(d, w, N_CTA, Bhat, N)
    assert _read(d, "status.i32", np.int32)[0] == 0

    s_h = s.numpy()
    idx = otg.retained_sets(s_h, ref["ntok"][0], N)
    kept = _read(d, "kept.i32", np.int32, (w.batch, w.H, Nmax))
    for b in range(w.batch):
        for h in range(w.H):
            n = int(ref["ntok"][0][b, h])
            assert np.array_equal(kept[b, h, :n], idx[b][h]), (b, h)
    out_ref, lse_ref = otg.decode_layer(q.float().numpy(), K.float().numpy(), V.float().numpy(), idx,
                                        1.0 / math.sqrt(w.d))
    bits = _read(d, "out.u16", np.uint16, (w.batch, w.H_q, w.d)).astype(np.uint32) << 16
    out = bits.view(np.float32).astype(np.float64)
    lse = _read(d, "lse.f32", np.float32, (w.batch, w.H_q)).astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    diff = np.abs(out - out_ref)
    assert diff.max() <= OUT_MAX_ABS and diff.mean() <= OUT_MEAN_ABS, (diff.max(), diff.mean())
    assert np.abs(lse[fin] - lse_ref[fin]).max() <= LSE_MAX_ABS


@pytest.mark.gpu
def test_c_consumer_selects_pages_and_decodes_on_the_gpu(consumer, tmp_path):
    """The page-selection path from C: MinMax cache, Quest page scores and top-K pages
    (bit-exact page lists), then decode attention over the selected pages (tolerance)."""
    import torch
    from gpu_helpers import OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS
    from oracle import flexicache as ofx

    w = synth.workload(4, batch=3, N=400, L=1)
    K_sel, N_CTA = 10, 40
    P, n_pages = w.P, w.N // w.P
    d = str(tmp_path)
    scale = 1.0 / math.sqrt(w.d)
    with open(os.path.join(d, "sdims"), "w") as f:
        f.write(f"{w.batch} {w.H} {w.H_q} {w.d} {w.N} {P} {K_sel} {N_CTA} {scale!r}\n")
    Kt, Vt = synth.keys_values(w, 0, "cpu")
    q = synth.queries(w, 0, "cpu")
    for name, t in (("K.u16", Kt), ("V.u16", Vt), ("q.u16", q)):
        t.contiguous().view(torch.int16).numpy().tofile(os.path.join(d, name))
    r = subprocess.run([consumer, d, "sparse"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert _read(d, "status.i32", np.int32)[0] == 0

    K_h, V_h, q_h = Kt.float().numpy(), Vt.float().numpy(), q.float().numpy()
    mn = np.zeros((w.batch, w.H, n_pages, w.d), np.float32)
    mx = np.zeros_like(mn)
    for b in range(w.batch):
        for h in range(w.H):
            mn[b, h], mx[b, h] = ofx.page_minmax(K_h[b, h], P)
    sel_ref = ofx.select_pages(q_h, mn, mx, K_sel)
    assert np.array_equal(_read(d, "sel.i32", np.int32, (w.batch, w.H, K_sel)), sel_ref)

    bits = _read(d, "out.u16", np.uint16, (w.batch, w.H_q, w.d)).astype(np.uint32) << 16
    out = bits.view(np.float32).astype(np.float64)
    lse = _read(d, "lse.f32", np.float32, (w.batch, w.H_q)).astype(np.float64)
    ref_out = np.zeros((w.batch, w.H_q, w.d))
    ref_lse = np.zeros((w.batch, w.H_q))
    for b in range(w.batch):
        for j in range(w.H_q):
            h = j // w.g
            tok = ofx.page_tokens(sel_ref[b, h], P, w.N)
            ref_out[b, j], ref_lse[b, j] = otg.attention(q_h[b, j], K_h[b, h][tok], V_h[b, h][tok], scale)
    diff = np.abs(out - ref_out)
    assert diff.max() <= OUT_MAX_ABS and diff.mean() <= OUT_MEAN_ABS, (diff.max(), diff.mean())
    assert np.abs(lse - ref_lse).max() <= LSE_MAX_ABS
