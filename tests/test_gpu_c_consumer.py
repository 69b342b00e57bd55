"""A plain C99 program as the library's user on the GPU: it owns the device
memory (cudaMalloc through the CUDA runtime's C API), sizes the workspaces,
and runs the fused forward and backward through include/lmhead.h alone. Its
outputs must carry the same bits as the same calls through the Python binding,
and match the fp64 oracle within the stated tolerances."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (ATOL_LOGPROB, RTOL_FROB_GRAD, f64, fused_case, max_abs, rel_frob, to_dev,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "lmhead.h"

/* argv: dir T H V inv_temperature; inputs and outputs are raw files in dir */
static void* slurp(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  FILE* f;
  void* p = malloc(bytes);
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "rb");
  if (!f || !p || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %s\n", path);
    exit(2);
  }
  fclose(f);
  return p;
}

static void spill(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  FILE* f;
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "wb");
  if (!f || fwrite(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    exit(2);
  }
  fclose(f);
}

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) exit(3);
  if (host && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) exit(3);
  return d;
}

#define TRY(call)                                                     \
  do {                                                                \
    int rc_ = (call);                                                 \
    if (rc_ != LMH_OK) {                                              \
      fprintf(stderr, "%s: %d %s\n", #call, rc_, lmhead_last_error_string()); \
      return 4;                                                       \
    }                                                                 \
  } while (0)

int main(int argc, char** argv) {
  const char* dir;
  int64_t T, H, V;
  float s;
  size_t hb, wb, ws_f, ws_b;
  void *hidden, *weight, *labels, *grad, *lp, *ent, *lse, *gh, *gw, *wsf, *wsb;
  void *h_lp, *h_ent, *h_lse, *h_gh, *h_gw;
  if (argc != 6) return 1;
  dir = argv[1];
  T = atoll(argv[2]);
  H = atoll(argv[3]);
  V = atoll(argv[4]);
  s = (float)atof(argv[5]);
  hb = (size_t)(T * H) * 2;
  wb = (size_t)(V * H) * 2;
  hidden = dev_copy(slurp(dir, "hidden.bin", hb), hb);
  weight = dev_copy(slurp(dir, "weight.bin", wb), wb);
  labels = dev_copy(slurp(dir, "labels.bin", (size_t)T * 4), (size_t)T * 4);
  grad = dev_copy(slurp(dir, "grad.bin", (size_t)T * 4), (size_t)T * 4);
  lp = dev_copy(NULL, (size_t)T * 4);
  ent = dev_copy(NULL, (size_t)T * 4);
  lse = dev_copy(NULL, (size_t)T * 4);
  gh = dev_copy(NULL, hb);
  gw = dev_copy(NULL, (size_t)(V * H) * 4);
  ws_f = lmhead_workspace_size(LMH_OP_FWD, T, H, V);
  ws_b = lmhead_workspace_size(LMH_OP_BWD, T, H, V);
  wsf = dev_copy(NULL, ws_f);
  wsb = dev_copy(NULL, ws_b);
  TRY(lmhead_logprob_fwd(hidden, weight, labels, T, H, V, s, lp, ent, lse, wsf, ws_f, NULL));
  TRY(lmhead_logprob_bwd(hidden, weight, labels, grad, lse, T, H, V, s, gh, gw, wsb, ws_b, NULL));
  if (cudaDeviceSynchronize() != cudaSuccess) return 5;
  {
    unsigned bits = 0;
    TRY(lmhead_device_status(NULL, &bits));
    if (bits != 0) return 6;
  }
  h_lp = malloc((size_t)T * 4);
  h_ent = malloc((size_t)T * 4);
  h_lse = malloc((size_t)T * 4);
  h_gh = malloc(hb);
  h_gw = malloc((size_t)(V * H) * 4);
  cudaMemcpy(h_lp, lp, (size_t)T * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_ent, ent, (size_t)T * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_lse, lse, (size_t)T * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_gh, gh, hb, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_gw, gw, (size_t)(V * H) * 4, cudaMemcpyDeviceToHost);
  spill(dir, "lp.bin", h_lp, (size_t)T * 4);
  spill(dir, "ent.bin", h_ent, (size_t)T * 4);
  spill(dir, "lse.bin", h_lse, (size_t)T * 4);
  spill(dir, "gh.bin", h_gh, hb);
  spill(dir, "gw.bin", h_gw, (size_t)(V * H) * 4);
  printf("ok\n");
  return 0;
}
"""


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    if not os.path.exists(os.path.join(home, "include", "cuda_runtime_api.h")):
        pytest.skip("CUDA runtime headers not found")
    return home


def test_c_program_forward_backward_matches_binding_and_oracle(tmp_path):
    import torch

    import invariant_lm_head_gb300 as lmh

    libdir = os.path.dirname(str(lmh.build()))
    cuda = _cuda_home()
    cc = shutil.which("gcc")
    if not cc:
        pytest.skip("gcc not found")
    src = tmp_path / "consumer.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "consumer"
    libcuda = os.path.join(cuda, "lib64")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", f"-I{INCLUDE}",
                        f"-I{cuda}/include", str(src), f"-L{libdir}", "-llmhead",
                        f"-L{libcuda}", "-lcudart", f"-Wl,-rpath,{libdir}",
                        f"-Wl,-rpath,{libcuda}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    T, H, V = 300, 264, 5000
    s = W.f32(1.0 / 0.7)
    hidden, weight, labels, grad = fused_case(61, T, H, V, w_std=0.05, oov=((5, -100),))
    np.ascontiguousarray(hidden).tofile(tmp_path / "hidden.bin")
    np.ascontiguousarray(weight).tofile(tmp_path / "weight.bin")
    np.ascontiguousarray(labels, dtype=np.int32).tofile(tmp_path / "labels.bin")
    np.ascontiguousarray(grad, dtype=np.float32).tofile(tmp_path / "grad.bin")
    r = subprocess.run([str(exe), str(tmp_path), str(T), str(H), str(V), repr(float(s))],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
    c_lp = np.fromfile(tmp_path / "lp.bin", dtype=np.float32)
    c_ent = np.fromfile(tmp_path / "ent.bin", dtype=np.float32)
    c_lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32)
    c_gh = np.fromfile(tmp_path / "gh.bin", dtype=np.uint16).reshape(T, H)
    c_gw = np.fromfile(tmp_path / "gw.bin", dtype=np.float32).reshape(V, H)

    # the same calls through the Python binding: the same bits
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    gh, gw = lmh.lmhead_logprob_bwd(h, w, lab, g, s, lse=lse)
    torch.cuda.synchronize()
    for c_val, py in ((c_lp, lp), (c_ent, ent), (c_lse, lse), (c_gw, gw)):
        assert np.array_equal(c_val.view(np.int32), py.cpu().numpy().view(np.int32))
    assert np.array_equal(c_gh, gh.cpu().view(torch.int16).numpy().view(np.uint16))

    # and the oracle within the stated tolerances
    rlp, rent, rlse = oracle.fused_forward(f64(hidden), f64(weight), labels, s)
    assert max_abs(c_lp, rlp) < ATOL_LOGPROB
    assert max_abs(c_ent, rent) < ATOL_LOGPROB
    assert max_abs(c_lse, rlse) < ATOL_LOGPROB
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, s)
    assert rel_frob(W.bf16_bits_to_f32(c_gh), rgh) < RTOL_FROB_GRAD
    assert rel_frob(c_gw, rgw) < RTOL_FROB_GRAD
