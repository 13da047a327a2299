"""The boundary from C: ``include/mhcpb.h`` compiles as strict C99 and as
C++17 (-Wall -Wextra -Werror -pedantic), and a C program linked against
``libmhcpb.so`` gets the documented host-side answers, all of which come
before any CUDA call, so no GPU is needed (the cuDNN frontend page "DSv4.1
mHC projection/RMS backward", "Requirements and tensor contract": allow_tf32
must be passed explicitly, other shapes are rejected)."""
import os
import shutil
import subprocess

import pytest

from rms_backward_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mhcpb.h"

/* each failed expectation exits with its own code */
#define EXPECT(n, cond) do { if (!(cond)) return (n); } while (0)

int main(void) {
    mhcpb_plan_t plan = NULL;
    size_t bytes = 1;
    int64_t value = 0;
    float f = 0.f;
    EXPECT(1, mhcpb_plan_create(&plan, 100, 512, 0, 0u) == MHCPB_ERR_TF32_NOT_ALLOWED);
    EXPECT(2, mhcpb_plan_create(&plan, -1, 512, 0, MHCPB_ALLOW_TF32) == MHCPB_ERR_UNSUPPORTED_SHAPE);
    EXPECT(3, mhcpb_plan_create(&plan, 100, 12, 0, MHCPB_ALLOW_TF32) == MHCPB_ERR_UNSUPPORTED_SHAPE);
    EXPECT(4, mhcpb_plan_create(&plan, (int64_t)MHCPB_MAX_T + 1, 512, 0, MHCPB_ALLOW_TF32) ==
              MHCPB_ERR_UNSUPPORTED_SHAPE);
    EXPECT(5, mhcpb_plan_create(NULL, 100, 512, 0, MHCPB_ALLOW_TF32) == MHCPB_ERR_INVALID_ARG);
    EXPECT(6, plan == NULL);
    EXPECT(7, mhcpb_workspace_bytes(NULL, &bytes) == MHCPB_ERR_INVALID_ARG);
    EXPECT(8, mhcpb_plan_query(NULL, 0, &value) == MHCPB_ERR_INVALID_ARG);
    EXPECT(9, mhcpb_destroy(NULL) == MHCPB_OK);
    /* the gate calls check the shape before anything else */
    EXPECT(10, mhcpb_gate_forward(-1, 20, &f, &f, &f, &f, &f, NULL) == MHCPB_ERR_UNSUPPORTED_SHAPE);
    EXPECT(11, mhcpb_gate_forward(4, MHCPB_GATE_MAX_ITER + 1, &f, &f, &f, &f, &f, NULL) ==
               MHCPB_ERR_UNSUPPORTED_SHAPE);
    EXPECT(12, strlen(mhcpb_status_string(MHCPB_OK)) > 0);
    printf("%s\n%s\n", mhcpb_status_string(MHCPB_ERR_TF32_NOT_ALLOWED),
           mhcpb_status_string(MHCPB_ERR_UNSUPPORTED_SHAPE));
    return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    if not os.path.exists(abi.LIB_PATH):
        from rms_backward_gb300 import build
        try:
            build.build()
        except RuntimeError as e:  # pragma: no cover
            pytest.skip(f"cannot build libmhcpb.so here: {e}")
    return os.path.dirname(abi.LIB_PATH)


def _compiler(name):
    cc = shutil.which(name)
    if cc is None:
        pytest.skip(f"{name} not found")
    return cc


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_strictly(tmp_path, lang, std):
    cc = _compiler("gcc" if lang == "c" else "g++")
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "mhcpb.h"\nint mhcpb_header_only_check;\n')
    subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, "-c", str(src),
                    "-o", str(tmp_path / "h.o")], check=True, capture_output=True, text=True)


def test_c_program_links_and_gets_the_documented_rejections(tmp_path, libdir):
    cc = _compiler("gcc")
    src = tmp_path / "consumer.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "consumer"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src),
                    "-L", libdir, "-lmhcpb", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, f"expectation {run.returncode} failed: {run.stdout} {run.stderr}"
    lines = run.stdout.strip().splitlines()
    assert lines == [abi.status_string(abi.MHCPB_ERR_TF32_NOT_ALLOWED),
                     abi.status_string(abi.MHCPB_ERR_UNSUPPORTED_SHAPE)]
