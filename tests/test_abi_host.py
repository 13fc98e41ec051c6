"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/hcr.h declares, and rejects bad create arguments on the host before
any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from kv_cache_restoration_gb300 import binding   # built at session start
    return binding


def declared_functions():
    with open(os.path.join(ROOT, "include", "hcr.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hcr_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("hcr_create", "hcr_restore", "hcr_destroy", "hcr_workspace_bytes",
              "hcr_check_device_error", "hcr_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(B.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(B):
    for s in range(8):
        assert B.hcr_status_string(s).startswith("HCR_")
    assert "unknown" in B.hcr_status_string(99)


def _dims(B, **kw):
    from kv_cache_restoration_gb300 import make_dims
    d = make_dims(2, 256, 4, 4, 64, max_position=128)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


FAKE = [0x1000, 0x2000]   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("field,value,status", [
    ("n_layers", 0, 1), ("d_model", 100, 1), ("d_model", 0, 1), ("n_kv_heads", 0, 1),
    ("n_heads", 6, 1), ("head_dim", 96, 2), ("norm", 5, 1), ("norm_eps", -1.0, 1),
    ("rope", 3, 1), ("rope_theta", 0.0, 1), ("max_position", 0, 1), ("dtype", 7, 1),
])
def test_create_rejects_bad_dims(B, field, value, status):
    st, h = B.hcr_create(_dims(B, **{field: value}), FAKE, None, FAKE, FAKE, check=False)
    assert st == status and h is None
    assert B.hcr_last_error()


def test_create_rejects_bad_pointers(B):
    d = _dims(B)
    assert B.hcr_create(d, None, None, FAKE, FAKE, check=False)[0] == B.HCR_ERR_INVALID_ARG
    assert B.hcr_create(d, FAKE, FAKE, FAKE, FAKE, check=False)[0] == B.HCR_ERR_INVALID_ARG
    assert B.hcr_create(d, [0x1000, 0], None, FAKE, FAKE, check=False)[0] == \
        B.HCR_ERR_INVALID_ARG
    assert B.hcr_create(d, FAKE, None, FAKE, FAKE, FAKE, FAKE, check=False)[0] == \
        B.HCR_ERR_INVALID_ARG
    ln = _dims(B, norm=B.HCR_NORM_LAYER)
    assert B.hcr_create(ln, FAKE, None, FAKE, FAKE, check=False)[0] == B.HCR_ERR_INVALID_ARG
    bias = _dims(B, has_kv_bias=1)
    assert B.hcr_create(bias, FAKE, None, FAKE, FAKE, check=False)[0] == B.HCR_ERR_INVALID_ARG


def test_null_handle_calls(B):
    assert B.hcr_workspace_bytes(None, 10, 1) == 0
    assert B.hcr_num_sms(None) == 0
    B.hcr_destroy(None)
    st = B.hcr_restore(None, None, 0, 1, 1, 1, None, None, None, 1, None, None, None, None, 0,
                       check=False)
    assert st == B.HCR_ERR_INVALID_ARG
    assert B.hcr_check_device_error(None)[0] == B.HCR_ERR_INVALID_ARG


C_CONSUMER = r"""
/* A plain C11 caller of the boundary: no C++, no CUDA headers. */
#include <stdio.h>
#include <string.h>
#include "hcr.h"

static int expect(int cond, const char* what) {
  if (!cond) fprintf(stderr, "failed: %s (last error: %s)\n", what, hcr_last_error());
  return cond ? 0 : 1;
}

int main(void) {
  int bad = 0;
  hcr_handle* h = NULL;
  hcr_model_dims d;
  memset(&d, 0, sizeof d);
  d.n_layers = 2; d.d_model = 256; d.n_heads = 4; d.n_kv_heads = 4; d.head_dim = 96;
  d.norm = HCR_NORM_RMS; d.norm_eps = 1e-5f; d.rope = HCR_ROPE_ROTATE_HALF;
  d.rope_theta = 10000.f; d.max_position = 128; d.dtype = HCR_DTYPE_BF16;
  bad += expect(hcr_create(NULL, NULL, NULL, NULL, NULL, NULL, NULL, &h) ==
                HCR_ERR_INVALID_ARG && h == NULL, "create without dims");
  bad += expect(hcr_create(&d, NULL, NULL, NULL, NULL, NULL, NULL, &h) != HCR_OK && h == NULL,
                "create with head_dim 96");
  bad += expect(strlen(hcr_last_error()) > 0, "last error names the failure");
  bad += expect(strcmp(hcr_status_string(HCR_OK), "HCR_OK") == 0, "status string");
  bad += expect(hcr_restore(NULL, NULL, 0, 1, 1, 1, NULL, NULL, NULL, 1, NULL, NULL, NULL, NULL,
                            0, NULL) == HCR_ERR_INVALID_ARG, "restore without a handle");
  hcr_destroy(NULL);
  if (!bad) printf("c consumer ok\n");
  return bad;
}
"""


def test_plain_c_consumer_compiles_links_and_runs(B, tmp_path):
    """include/hcr.h is a C header: a C11 program (gcc -std=c11 -pedantic,
    warnings as errors) includes it, links libhcr.so and calls the host-side
    paths that need no GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src, exe = tmp_path / "consumer.c", tmp_path / "consumer"
    src.write_text(C_CONSUMER)
    libdir = os.path.dirname(B.LIB)
    cmd = [gcc, "-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", libdir, "-l:" + os.path.basename(B.LIB), "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c consumer ok" in r.stdout, (r.stdout, r.stderr)
