"""The C ABI from plain C: a C program (tests/c_abi/hc_c_client.c), compiled
against include/hc.h and linked to libhc.so, runs encode, table, fetch and
the CRC-32 of the wire on cudaMalloc'd buffers, and asks for the default
selection size; its outputs are compared with the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from tests import parity
from oracle.numerics import round_to

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    import __graft_entry__
    lib = __graft_entry__.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("c_client") / "hc_c_client")
    cuda = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))
    cmd = [shutil.which("gcc") or "cc", "-O2", "-std=c99", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi", "hc_c_client.c"),
           "-o", exe, "-L", libdir, "-lhc", "-Wl,-rpath," + libdir,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_matches_the_oracle(client, tmp_path):
    c = parity.random_case(91, L=2, H=3, d=128, B=16, nb=5, src_fmt="f16", out_fmt="f32",
                           pairing="half_split", ragged=True)
    dm_vals, dm_idx = np.unique(c.delta_m, return_inverse=True)
    S_src, S_dst = c.src_k.shape[1], c.num_dst_slots
    init = np.full((c.L, S_dst, c.B, c.H, c.d), parity.SENTINEL, np.float32)
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(np.array([c.L, c.H, c.d, c.B, S_src, S_dst, len(c.src_slots), len(dm_vals)],
                         "<i4").tobytes())
        f.write(np.array([c.rope_base], "<f8").tobytes())
        f.write(c.src_k.astype("<f2").tobytes())
        f.write(c.src_v.astype("<f2").tobytes())
        for a in (c.src_slots, c.dst_slots, c.n_valid, dm_idx, dm_vals):
            f.write(np.asarray(a, "<i4").tobytes())
        f.write(init.tobytes())
    out = tmp_path / "out.bin"
    r = subprocess.run([client, str(inp), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = np.fromfile(out, np.uint8)
    nb, L, H, B, d = len(c.src_slots), c.L, c.H, c.B, c.d
    n_codes, n_scales, n_dst = L * nb * 2 * H * B * d, L * nb * 2 * H, L * S_dst * B * H * d
    codes = raw[:n_codes].reshape(L, nb, 2, H, B, d)
    o = n_codes
    scales = raw[o:o + 4 * n_scales].view("<f4").reshape(L, nb, 2, H)
    o += 4 * n_scales
    k = raw[o:o + 4 * n_dst].view("<f4").reshape(L, S_dst, B, H, d)
    o += 4 * n_dst
    v = raw[o:o + 4 * n_dst].view("<f4").reshape(L, S_dst, B, H, d)
    o += 4 * n_dst
    err = int(raw[o:o + 4].view("<i4")[0])
    o += 4
    crc = raw[o:o + 4 * L * nb].view("<u4")
    o += 4 * L * nb
    k_default = int(raw[o:o + 4].view("<i4")[0])
    assert o + 4 == raw.size
    want = parity.oracle_run(c, "fp8")
    assert err == 0
    assert np.array_equal(codes, want["codes"])
    assert np.array_equal(scales.astype(np.float64), want["scales"])
    rep = parity.compare_outputs(c, "fp8", {"k": k.astype(np.float64), "v": v.astype(np.float64)},
                                 want)
    assert rep["k_ok"] and rep["v_ok"] and rep["k_untouched_ok"] and rep["v_untouched_ok"], rep
    from oracle import blend, crc32 as ocrc
    a = want["codes"].reshape(L * nb, -1)
    b = want["scales"].astype("<f4").reshape(L * nb, -1).view(np.uint8)
    assert np.array_equal(crc, ocrc.crc32_units(a, a.shape[1], a.shape[1], L * nb, b, b.shape[1],
                                                b.shape[1]))
    assert k_default == blend.default_k(1408) == 212
