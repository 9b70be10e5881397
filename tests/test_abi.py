"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/santa.h declares, and rejects bad arguments on
the host (before any CUDA call) with the documented status codes."""
import ctypes
import os
import subprocess

import pytest

import stochastic_sparse_decode_split_gb300 as santa
from stochastic_sparse_decode_split_gb300 import build as santa_build

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    santa_build.build()
    return santa.library()


def params(**kw):
    p = santa.Params()
    p.batch, p.n_q_heads, p.n_kv_heads, p.head_dim = 1, 32, 8, 128
    p.dtype, p.nk, p.S, p.scale, p.seed, p.step = 0, 32768, 256, 0.0, 0, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_every_declared_symbol_is_exported(lib):
    names = santa.exported_symbols()
    assert {"santa_decode", "santa_dense_decode", "santa_workspace_size", "santa_get_error"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", santa_build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in names:
        assert hasattr(lib, n)


def test_device_error_bits_match_the_header():
    """The binding's DEVERR_* constants are the header's SANTA_DEVERR_* values
    (the library itself static_asserts the header against the kernels)."""
    import re
    hdr = open(os.path.join(santa_build.ROOT, "include", "santa.h")).read()
    found = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define SANTA_DEVERR_(\w+) (\d+)", hdr)}
    assert found == {"NK_BOUND": santa.DEVERR_NK_BOUND, "S_RANGE": santa.DEVERR_S_RANGE,
                     "EMPTY": santa.DEVERR_EMPTY, "TIMEOUT": santa.DEVERR_TIMEOUT}
    assert sorted(found.values()) == [1, 2, 4, 8]


def test_status_strings_and_version(lib):
    for code in range(6):
        assert lib.santa_status_string(code)
    assert lib.santa_status_string(99) == b"unknown status"
    assert lib.santa_version() >= 100


def test_workspace_size_valid_and_invalid(lib):
    p = params()
    n = santa.workspace_size(p)
    # stash alone is B*H*nk fp32
    assert n >= 32 * 32768 * 4
    assert n % 256 == 0
    assert santa.workspace_size(params(n_kv_heads=5)) == 0          # H % H_kv != 0
    assert santa.workspace_size(params(head_dim=96)) == 0           # unsupported head_dim
    assert santa.workspace_size(params(S=0)) == 0
    assert santa.workspace_size(params(S=4097)) == 0
    assert santa.workspace_size(params(nk=0)) == 0
    assert santa.workspace_size(params(nk=(1 << 21) + 1)) == 0
    assert santa.workspace_size(params(n_q_heads=72, n_kv_heads=8)) == 0   # group 9 > 8
    assert santa.dense_workspace_size(params(S=0)) > 0                   # dense ignores S
    lay = santa.workspace_layout(p)
    assert lay["chunks"] == 32768 // 16
    offs = sorted(lay[k] for k in ("stash", "tile_max", "tile_sum", "prefix", "thresh", "head_max"))
    assert offs[0] >= 256 and offs[-1] < n and all(o % 256 == 0 for o in offs)


def _decode(lib, p, variant=2, q=256, K=256, V=256, out=256, ws=None, nbytes=0):
    vp = ctypes.c_void_p
    return lib.santa_decode(ctypes.byref(p), variant, vp(q), vp(K), vp(V), vp(out), vp(ws), nbytes, None, None)


def test_host_validation_statuses(lib):
    """Every case below fails a host check that precedes all CUDA calls."""
    good = params()
    n = santa.workspace_size(good)
    assert _decode(lib, params(n_kv_heads=3)) == INVALID
    assert _decode(lib, params(batch=0)) == INVALID
    assert _decode(lib, params(S=0)) == INVALID
    assert _decode(lib, params(head_dim=80)) == UNSUPPORTED
    assert _decode(lib, params(dtype=7)) == UNSUPPORTED
    assert _decode(lib, params(scale=float("nan"))) == INVALID
    assert _decode(lib, good, variant=3) == INVALID
    assert _decode(lib, good, q=0) == INVALID                     # NULL q
    assert _decode(lib, good, K=264) == INVALID                   # K not 16-byte aligned
    assert _decode(lib, good, ws=None, nbytes=n) == WORKSPACE     # no workspace
    assert _decode(lib, good, ws=512 + 16, nbytes=n) == WORKSPACE  # misaligned workspace
    assert _decode(lib, good, ws=512, nbytes=n - 256) == WORKSPACE  # too small
    vp = ctypes.c_void_p
    assert lib.santa_decode_with_uniforms(ctypes.byref(good), 2, vp(256), vp(256), vp(256), None, vp(256), vp(512),
                                          n, None, None) == INVALID
    assert lib.santa_dense_decode(ctypes.byref(params(head_dim=32)), vp(256), vp(256), vp(256), vp(256), vp(512),
                                  1 << 30, None) == UNSUPPORTED
    assert lib.santa_workspace_init(None, 1024, None) == WORKSPACE
    assert lib.santa_get_error(vp(512 + 8), None, None) == WORKSPACE
    # host-resident K/V: parameters and NULL buffers are refused before the pointer queries
    assert lib.santa_decode_host_kv(ctypes.byref(params(batch=0)), 2, vp(256), vp(256), vp(256), vp(256), vp(512),
                                    n, None, None) == INVALID
    assert lib.santa_decode_host_kv(ctypes.byref(good), 2, vp(256), None, vp(256), vp(256), vp(512), n, None,
                                    None) == INVALID
    assert lib.santa_decode_host_kv(ctypes.byref(good), 2, vp(256), vp(256), None, vp(256), vp(512), n, None,
                                    None) == INVALID


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    K = torch.zeros(16, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        santa.santa_decode(q, K, K, S=4)


def test_host_validation_of_the_tile_samplers_bernoulli_and_helpers(lib):
    """The other entry points' argument checks, all before any CUDA call."""
    vp = ctypes.c_void_p
    good = params()
    n_t = santa.tiled_workspace_size(good, "prop", 256)
    assert n_t > santa.workspace_size(good)
    assert santa.tiled_max_draws(good, "prop", 256) == good.S
    assert santa.tiled_max_draws(good, "flash", 256) == good.S + 32768 // 256
    for L in (0, 8, 24, 2048):
        assert santa.tiled_workspace_size(good, "prop", L) == 0
    assert lib.santa_tiled_workspace_size(ctypes.byref(good), 2, 256) == 0           # no third sampler

    def tiled(p=good, sampler=0, L=256, q=256, ws=512, nbytes=n_t):
        return lib.santa_decode_tiled(ctypes.byref(p), sampler, L, vp(q), vp(256), vp(256), vp(256), vp(ws), nbytes,
                                      None, None)
    assert tiled(L=40) == INVALID
    assert tiled(sampler=5) == INVALID
    assert tiled(p=params(S=0)) == INVALID
    assert tiled(q=0) == INVALID
    assert tiled(nbytes=n_t - 256) == WORKSPACE

    n_b = santa.bernoulli_workspace_size(good)
    assert n_b > santa.workspace_size(good)

    def bern(n=4, variant=2, ws=512, nbytes=n_b):
        return lib.santa_decode_bernoulli(ctypes.byref(good), variant, n, 1, vp(256), vp(256), vp(256), vp(256),
                                          vp(ws), nbytes, None, None, None)
    assert bern(n=0) == INVALID and bern(n=1025) == INVALID
    assert bern(variant=7) == INVALID
    assert bern(nbytes=n_b - 256) == WORKSPACE

    assert lib.santa_read_probe(None, 1024, vp(256), None) == INVALID
    assert lib.santa_read_probe(vp(256), 1000, vp(256), None) == INVALID               # not a multiple of 16
    assert lib.santa_read_probe(vp(264), 1024, vp(256), None) == INVALID               # not 16-byte aligned
    assert lib.santa_read_probe_sink_words() >= 2 * 512
    assert lib.santa_selftest_wait_timeout(None, 4096, 50_000_000, None) == WORKSPACE
    assert lib.santa_selftest_wait_timeout(vp(512), 4096, 10, None) == INVALID          # below 1 ms
    assert lib.santa_selftest_wait_timeout(vp(512), 4096, 3_000_000_000, None) == INVALID


C_CLIENT = r"""
#include <stdio.h>
#include "santa.h"
int main(void) {
  santa_params_t p = {0};
  p.batch = 1; p.n_q_heads = 32; p.n_kv_heads = 8; p.head_dim = 128;
  p.dtype = SANTA_BF16; p.nk = 32768; p.S = 256;
  size_t n = santa_workspace_size(&p);
  p.n_kv_heads = 3;   /* 32 query heads do not split into 3 groups */
  santa_status_t st = santa_decode(&p, SANTA_SYSTEMATIC, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL);
  printf("%d %zu %d %s\n", santa_version(), n, (int)st, santa_status_string(st));
  return n == 0 || st != SANTA_ERR_INVALID_ARG;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/santa.h compiles as strict C99 (gcc -pedantic -Werror) and a C
    program links against the library and calls its host-side functions."""
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = santa_build.BUILD
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                    os.path.join(santa_build.ROOT, "include"), str(src), "-o", str(exe), "-L", libdir,
                    "-l:libsanta.so", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert int(out[0]) >= 100 and int(out[1]) == santa.workspace_size(params()) and int(out[2]) == INVALID
