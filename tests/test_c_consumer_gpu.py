"""A plain C program restores a cache through the C ABI alone (GPU).

The test writes a small ragged case's inputs (hidden states, per-layer
weights, request metadata) to files; a C11 program, compiled here with gcc
against include/hcr.h and the CUDA runtime, loads them into device memory,
creates a handle, restores, checks the device error word and writes both
caches back.  They must equal, bit for bit, the caches the Python binding
produces from the same inputs (both start from the same sentinel-filled
caches), and the binding's result is checked against the oracle.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from tests import harness as Hn
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = Workload("c-abi", ModelShape("cabi", 2, 256, 4, 4, 64), (77, 130, 0, 5), (3, 0, 9, 200),
             block_order="shuffled", spare_blocks=2)

PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime.h>
#include "hcr.h"

static const char* g_dir;

static void* load(const char* name, size_t* bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", g_dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(3); }
  fseek(f, 0, SEEK_END);
  long n = ftell(f);
  fseek(f, 0, SEEK_SET);
  void* p = malloc((size_t)n > 0 ? (size_t)n : 1);
  if (fread(p, 1, (size_t)n, f) != (size_t)n) { fprintf(stderr, "short read %s\n", path); exit(3); }
  fclose(f);
  if (bytes) *bytes = (size_t)n;
  return p;
}

static void* to_device(const char* name, size_t* bytes) {
  size_t n = 0;
  void* h = load(name, &n);
  if (bytes) *bytes = n;
  void* d = NULL;
  if (cudaMalloc(&d, n > 0 ? n : 16) != cudaSuccess) exit(4);
  if (n && cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) exit(4);
  free(h);
  return d;
}

static void save(const char* name, const void* dev, size_t n) {
  char path[4096];
  void* h = malloc(n);
  snprintf(path, sizeof path, "%s/%s", g_dir, name);
  if (cudaMemcpy(h, dev, n, cudaMemcpyDeviceToHost) != cudaSuccess) exit(4);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(h, 1, n, f) != n) exit(3);
  fclose(f);
  free(h);
}

int main(int argc, char** argv) {
  enum { MAX_LAYERS = 8 };
  const void* gamma[MAX_LAYERS];
  const void* w_k[MAX_LAYERS];
  const void* w_v[MAX_LAYERS];
  int32_t* m;
  float* f;
  hcr_model_dims dims;
  hcr_cache_layout layout;
  hcr_handle* h = NULL;
  hcr_status st;
  int32_t L, T, R, max_blocks, l;
  size_t ws_bytes, cache_bytes;
  void *hidden, *cu, *start, *table, *ws, *kc, *vc;
  uint32_t flags = 0;
  char name[64];

  if (argc != 2) return 2;
  g_dir = argv[1];
  /* meta: n_layers d_model n_heads n_kv_heads head_dim norm rope max_position dtype
           has_kv_bias n_tokens n_req num_blocks block_size max_blocks; floats: eps theta */
  m = (int32_t*)load("meta.i32", NULL);
  f = (float*)load("meta.f32", NULL);
  memset(&dims, 0, sizeof dims);
  dims.n_layers = m[0]; dims.d_model = m[1]; dims.n_heads = m[2]; dims.n_kv_heads = m[3];
  dims.head_dim = m[4]; dims.norm = m[5]; dims.rope = m[6]; dims.max_position = m[7];
  dims.dtype = m[8]; dims.has_kv_bias = m[9]; dims.norm_eps = f[0]; dims.rope_theta = f[1];
  L = m[0]; T = m[10]; R = m[11]; max_blocks = m[14];
  layout.num_blocks = m[12]; layout.block_size = m[13]; layout.layer_stride_elems = 0;
  if (L > MAX_LAYERS) return 2;
  for (l = 0; l < L; ++l) {
    snprintf(name, sizeof name, "gamma%d.bin", l); gamma[l] = to_device(name, NULL);
    snprintf(name, sizeof name, "wk%d.bin", l); w_k[l] = to_device(name, NULL);
    snprintf(name, sizeof name, "wv%d.bin", l); w_v[l] = to_device(name, NULL);
  }
  st = hcr_create(&dims, gamma, NULL, w_k, w_v, NULL, NULL, &h);
  if (st != HCR_OK) { fprintf(stderr, "create: %s\n", hcr_last_error()); return 10 + (int)st; }
  hidden = to_device("hidden.bin", NULL);
  cu = to_device("cu.i32", NULL);
  start = to_device("start.i32", NULL);
  table = to_device("table.i32", NULL);
  ws_bytes = hcr_workspace_bytes(h, T, L);
  if (cudaMalloc(&ws, ws_bytes) != cudaSuccess) return 4;
  /* the caches as they were before the restore (sentinel-filled) */
  kc = to_device("k0.bin", &cache_bytes);
  vc = to_device("v0.bin", NULL);
  if (cache_bytes != (size_t)L * layout.num_blocks * layout.block_size * dims.n_kv_heads *
                         dims.head_dim * 2)
    return 5;
  st = hcr_restore(h, hidden, 0, L, R, T, (const int32_t*)cu, (const int32_t*)start,
                   (const int32_t*)table, max_blocks, kc, vc, &layout, ws, ws_bytes, NULL);
  if (st != HCR_OK) { fprintf(stderr, "restore: %s\n", hcr_last_error()); return 20 + (int)st; }
  st = hcr_check_device_error(h, NULL, &flags);
  if (st != HCR_OK || flags) { fprintf(stderr, "device error %u\n", flags); return 30 + (int)st; }
  save("k.bin", kc, cache_bytes);
  save("v.bin", vc, cache_bytes);
  hcr_destroy(h);
  printf("c restore ok\n");
  return 0;
}
"""


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy()


def test_c_program_restores_like_the_binding(cuda_device, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from kv_cache_restoration_gb300 import binding as B
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    case = Hn.make_case(W, cuda_device)
    _bits(case.k_cache).tofile(tmp_path / "k0.bin")
    _bits(case.v_cache).tofile(tmp_path / "v0.bin")
    Hn.run(case)
    assert case.status == 0
    Hn.compare(case)

    lay = case.layout
    dims = Hn.dims_for(W)
    meta = [dims.n_layers, dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.norm,
            dims.rope, dims.max_position, dims.dtype, dims.has_kv_bias, W.n_tokens,
            int(case.start.numel()), lay.num_blocks, lay.block_size, lay.max_blocks]
    np.asarray(meta, np.int32).tofile(tmp_path / "meta.i32")
    np.asarray([dims.norm_eps, dims.rope_theta], np.float32).tofile(tmp_path / "meta.f32")
    _bits(case.hidden).tofile(tmp_path / "hidden.bin")
    for l, p in enumerate(case.params):
        _bits(p.gamma).tofile(tmp_path / f"gamma{l}.bin")
        _bits(p.w_k).tofile(tmp_path / f"wk{l}.bin")
        _bits(p.w_v).tofile(tmp_path / f"wv{l}.bin")
    for name, t in (("cu", case.cu), ("start", case.start), ("table", case.table)):
        t.to(torch.int32).cpu().numpy().tofile(tmp_path / f"{name}.i32")

    src, exe = tmp_path / "restore.c", tmp_path / "restore"
    src.write_text(PROGRAM)
    libdir = os.path.dirname(B.LIB)
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), str(src), "-o", str(exe),
           "-L", libdir, "-l:" + os.path.basename(B.LIB), "-Wl,-rpath," + libdir,
           "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "c restore ok" in r.stdout, (r.returncode, r.stdout, r.stderr)
    for name, ref in (("k.bin", case.k_cache), ("v.bin", case.v_cache)):
        got = np.fromfile(tmp_path / name, dtype=np.int16)
        want = _bits(ref).reshape(-1)
        assert got.shape == want.shape
        assert np.array_equal(got, want), f"{name}: {int((got != want).sum())} elements differ"
