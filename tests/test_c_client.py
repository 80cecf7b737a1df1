"""The C ABI from plain C: tests/c_client/decode_step.c is compiled with gcc
against include/pkv.h and the CUDA runtime (no Python, no torch in that
process), runs one decode step on device buffers it allocates itself, and
must return the same bits as the Python binding; both match the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from paged_kv_cache_loc_gb300 import build
from paged_kv_cache_loc_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))


@pytest.mark.gpu
def test_c_client_decode_step_matches_the_binding(tmp_path):
    import torch
    import paged_kv_cache_loc_gb300 as pkv
    lib = build.build()
    case = W.batched_decode(batch=8, lo=100, hi=1500, size=16384, seed=4242)
    meta = [case.k_buffer.shape[0], case.k_buffer.shape[1], case.n_kv_heads, case.head_dim,
            case.req_to_token.shape[0], case.req_to_token.shape[1], case.batch, case.n_heads,
            case.layer_id, case.max_len]
    (tmp_path / "meta.txt").write_text(" ".join(str(int(x)) for x in meta))
    for name in ("k_buffer", "v_buffer", "req_to_token", "req_pool_indices", "seq_lens", "kv_indptr",
                 "out_cache_loc", "q", "k_new", "v_new"):
        np.ascontiguousarray(getattr(case, name)).tofile(tmp_path / f"{name}.bin")
    exe = tmp_path / "decode_step"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(CUDA, "include"),
                           os.path.join(ROOT, "tests", "c_client", "decode_step.c"), "-o", str(exe),
                           lib, "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
                           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(CUDA, "lib64")])
    out = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    o_c = np.fromfile(tmp_path / "o.bin", np.uint16).reshape(case.q.shape)

    cache, q, kn, vn = W.upload(case)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 256)
    o = pkv.decode_step(cache, case.layer_id, kn, vn, q, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(W.host_of(o), o_c)
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    ref = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                        case.seq_lens, case.q, case.layer_id, kv_indptr=case.kv_indptr)
    err = np.abs(oracle.to_f64(o_c) - ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
