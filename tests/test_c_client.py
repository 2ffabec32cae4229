"""The boundary from plain C: a C99 program includes include/lightning_attn.h, links
liblightning_attn.so with gcc, and exercises the host-side part of the ABI (no GPU
needed: every call below is rejected or completed before anything is launched).
"""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include "lightning_attn.h"

#define CHECK(expr, want)                                                    \
    do {                                                                     \
        int got_ = (expr);                                                   \
        if (got_ != (want)) {                                                \
            printf("FAIL %s: got %d want %d\n", #expr, got_, (int)(want));   \
            return 1;                                                        \
        }                                                                    \
    } while (0)

int main(void) {
    /* fake, 16-byte aligned addresses that are never dereferenced */
    void* p[6] = {(void*)0x10000, (void*)0x20000, (void*)0x30000,
                  (void*)0x40000, (void*)0x50000, (void*)0x60000};
    float* st = (float*)0x70000;
    CHECK(la_version() >= 200, 1);
    CHECK(la_prefill(p[0], p[1], p[2], p[3], p[4], st, 1, 2, 16, 64), LA_ERR_UNSUPPORTED);
    CHECK(la_prefill(NULL, p[1], p[2], p[3], p[4], st, 1, 2, 16, 128), LA_ERR_INVALID_ARG);
    CHECK(la_decode_step(st, p[1], p[2], p[3], p[4], p[5], 0, 2, 128), LA_ERR_INVALID_ARG);
    CHECK(la_prefill_ex(p[0], p[1], p[2], p[3], p[4], st, NULL, NULL, 1, 2, 16, 128, LA_BF16,
                        1e-6f, 0x100u, NULL), LA_ERR_INVALID_ARG);
    CHECK(la_qkvg_projection(p[0], p[1], p[2], p[3], p[4], p[5], 16, 64, 1, 128,
                             LA_PROJ_SILU, NULL), LA_ERR_UNSUPPORTED);
    CHECK(la_softmax_attention(p[0], p[1], p[2], p[3], 1, 2, 16, 128, 1.0, NULL),
          LA_ERR_INVALID_ARG);
    {
        const int64_t cu[3] = {0, 5, 3};
        CHECK(la_prefill_varlen(p[0], p[1], p[2], p[3], p[4], st, cu, 2, 2, 128),
              LA_ERR_INVALID_ARG);
    }
    CHECK(la_decode_step_noalloc(st, p[1], p[2], p[3], p[4], p[5], 200, 128, 128, LA_BF16,
                                 1e-6f, NULL), LA_ERR_SCRATCH_LIMIT);
    CHECK(la_prefill_path(1, 1, 1, 128, LA_F32, 0), 1);
    printf("ok %s\n", la_status_string(LA_ERR_TIMEOUT));
    return 0;
}
"""


def test_c_program_links_and_calls_the_abi(tmp_path):
    from linear_attention_hybrid_fwd_b300 import build as la_build
    lib = la_build.build()
    src = tmp_path / "client.c"
    src.write_text(C_SRC)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-L", libdir, "-llightning_attn",
                           "-Wl,-rpath," + libdir, "-o", str(exe)])
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.startswith("ok ")
