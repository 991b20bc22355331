"""The C ABI used from plain C: tests/c/abi_client.c is compiled against
include/vcoll.h and linked to libvcoll.so.  Host mode runs anywhere; GPU
mode allreduces integer-valued buffers whose exact sums are known."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = "/usr/local/cuda"


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    from collective_reduction_virtual_gb300 import build
    lib = build.build()
    exe = str(tmp_path_factory.mktemp("c") / "abi_client")
    cc = shutil.which("gcc") or "cc"
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-o", exe, os.path.join(HERE, "c", "abi_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.dirname(lib) + "/libvcoll.so", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe, *args):
    r = subprocess.run([exe, *args], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    return [ln.split() for ln in r.stdout.splitlines()]


def test_c_client_host_mode(client):
    lines = _run(client)
    segs = [ln for ln in lines if ln[0] == "segment"]
    assert [(int(a), int(b)) for _, _, a, b in segs] == [oracle.segment(1003, 4, j) for j in range(4)]
    plan = [ln for ln in lines if ln[0] == "plan"][0]
    assert [int(v) for v in plan[1:]] == oracle.fuse_plan([10, 10, 10, 30, 2], oracle.F32, 100)
    d = {ln[0]: ln[1:] for ln in lines}
    assert d["bad_op"] == ["3"] and d["bad_type"] == ["2"] and d["bad_w"] == ["1"]
    assert d["empty"] == ["0"]
    assert " ".join(d["status"]) == "invalid reduction operation"


def _inputs():
    n, W = 1003, 4
    return [np.array([(i * 7 + u * 13) % 41 - 20 for i in range(n)], np.float32) for u in range(W)]


def _bits(lines, tag):
    out = {}
    for ln in lines:
        if ln[0] == tag:
            out.setdefault(int(ln[1]), []).append((int(ln[2]), int(ln[3], 16)))
    return {u: [b for _, b in sorted(v)] for u, v in out.items()}


@pytest.mark.gpu
def test_c_client_gpu_mode(client):
    lines = _run(client, "gpu")
    ins = _inputs()
    W = len(ins)
    ar = [a.view(np.uint32).tolist() for a in oracle.allreduce(ins, "sum", oracle.F32)]
    assert _bits(lines, "ag") == {u: ar[u] for u in range(W)}
    assert _bits(lines, "ar") == {u: ar[u] for u in range(W)}
    rsr = oracle.reduce_scatter(ins, "avg", oracle.F32, [1, 2, 0, 3])
    assert _bits(lines, "rsr") == {j: rsr[j].view(np.uint32).tolist() for j in range(W)}
    counts = [1003 - 353, 3, 350]
    offs = np.cumsum([0] + counts)
    tens = [[ins[u][offs[t]:offs[t + 1]] for t in range(3)] for u in range(W)]
    fb = oracle.fusion_allreduce(tens, counts, "sum", oracle.F32, 1 << 20)
    assert _bits(lines, "fb") == {u: np.concatenate(fb[u]).view(np.uint32).tolist()
                                  for u in range(W)}
    assert [ln for ln in lines if ln[0] == "fb_batches"] == [["fb_batches", "1"]]
