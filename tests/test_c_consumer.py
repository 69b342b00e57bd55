"""The boundary as a C program sees it: include/lmhead.h compiles as C99 and as
C++17 with every warning an error, a C program links against the in-tree
liblmhead.so, and its host-side calls (version, workspace sizes, argument
errors and their messages, empty batches) behave as the header states, with
no GPU and no kernel launched."""

import os
import shutil
import subprocess

import pytest

import invariant_lm_head_gb300 as lmh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "lmhead.h"

static int fails = 0;
#define CHECK(c)                                                      \
  do {                                                                \
    if (!(c)) {                                                       \
      fprintf(stderr, "failed at line %d: %s\n", __LINE__, #c);        \
      ++fails;                                                        \
    }                                                                 \
  } while (0)

/* never dereferenced: every call below fails validation, or has nothing to do */
#define FAKE(type, addr) ((type)(uintptr_t)(addr))

int main(void) {
  unsigned long long launches = lmhead_kernel_launches();
  float out[8];
  size_t fwd, bwd;
  int rc;

  CHECK(lmhead_abi_version() == 1);
  CHECK(lmhead_workspace_size(LMH_OP_LOGITS, 8192, 0, 152064) == 0);
  fwd = lmhead_workspace_size(LMH_OP_FWD, 16384, 3584, 152064);
  bwd = lmhead_workspace_size(LMH_OP_BWD, 16384, 3584, 152064);
  CHECK(fwd > 0 && fwd != SIZE_MAX);
  CHECK(bwd > fwd && bwd != SIZE_MAX);
  CHECK(lmhead_workspace_size(LMH_OP_FWD, LMH_MAX_DIM + 1, 256, 4096) == SIZE_MAX);
  CHECK(lmhead_workspace_size(7, 16, 256, 4096) == SIZE_MAX);

  /* a NULL input: refused with a message that names it */
  rc = lmhead_logprob_fwd(NULL, FAKE(const uint16_t*, 16), FAKE(const int32_t*, 16), 4, 256,
                          4096, 1.0f, out, NULL, NULL, FAKE(void*, 256), fwd, NULL);
  CHECK(rc == LMH_ERR_INVALID_ARG);
  CHECK(strstr(lmhead_last_error_string(), "hidden") != NULL);
  /* H not a multiple of 8, then a temperature that is not finite and positive */
  rc = lmhead_logprob_fwd(FAKE(const uint16_t*, 16), FAKE(const uint16_t*, 16),
                          FAKE(const int32_t*, 16), 4, 12, 4096, 1.0f, out, NULL, NULL,
                          FAKE(void*, 256), fwd, NULL);
  CHECK(rc == LMH_ERR_ALIGNMENT);
  rc = lmhead_logprob_fwd(FAKE(const uint16_t*, 16), FAKE(const uint16_t*, 16),
                          FAKE(const int32_t*, 16), 4, 256, 4096, -1.0f, out, NULL, NULL,
                          FAKE(void*, 256), fwd, NULL);
  CHECK(rc == LMH_ERR_INVALID_ARG);
  /* a workspace too small for the backward */
  rc = lmhead_logprob_bwd(FAKE(const uint16_t*, 16), FAKE(const uint16_t*, 16),
                          FAKE(const int32_t*, 16), FAKE(const float*, 16), NULL, 4, 256, 4096,
                          1.0f, FAKE(uint16_t*, 16), FAKE(float*, 16), FAKE(void*, 256), 16,
                          NULL);
  CHECK(rc == LMH_ERR_WORKSPACE);
  CHECK(strstr(lmhead_last_error_string(), "workspace") != NULL);
  /* the logits path with a misaligned logits pointer */
  rc = logprob_from_logits(FAKE(const uint16_t*, 24), FAKE(const int32_t*, 16), 4, 4096, 1.0f,
                           out, NULL, NULL, NULL);
  CHECK(rc == LMH_ERR_ALIGNMENT);
  /* an empty batch is a no-op, pointers may be NULL */
  rc = lmhead_logprob_fwd(NULL, FAKE(const uint16_t*, 16), NULL, 0, 256, 4096, 1.0f, NULL, NULL,
                          NULL, NULL, 0, NULL);
  CHECK(rc == LMH_OK);

  CHECK(lmhead_kernel_launches() == launches);
  if (!fails) printf("ok\n");
  return fails ? 1 : 0;
}
"""


def _compiler(name):
    path = shutil.which(name)
    if not path:
        pytest.skip(f"{name} not found")
    return path


@pytest.fixture(scope="module")
def libdir():
    return os.path.dirname(str(lmh.build()))


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_header_compiles_cleanly(tmp_path, lang):
    cc = _compiler("gcc" if lang == "c99" else "g++")
    src = tmp_path / ("h.c" if lang == "c99" else "h.cc")
    src.write_text('#include "lmhead.h"\nint lmhead_header_only(void) { return LMH_OK; }\n')
    r = subprocess.run([cc, f"-std={lang}", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        f"-I{INCLUDE}", "-c", str(src), "-o", str(tmp_path / "h.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_calls_the_library(tmp_path, libdir):
    cc = _compiler("gcc")
    src = tmp_path / "consumer.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "consumer"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", f"-I{INCLUDE}", str(src),
                        f"-L{libdir}", "-llmhead", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
