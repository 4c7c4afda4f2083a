"""The boundary as a C program sees it: `include/nvfp4.h` compiles as strict
C11 and as C++17 with every warning an error, and a plain C program linked
against libnvfp4.so gets the layout helpers, the argument checks and the
status strings without any Python or torch.  The program runs with every
GPU hidden, so a valid call reports NVFP4_ERR_DEVICE and nothing is
launched."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "nvfp4_precision_02_b300")

C_PROGRAM = r"""
#include "nvfp4.h"
#include <stdio.h>
#include <string.h>

static int fails = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #cond); ++fails; } } while (0)

int main(void) {
    /* layout helpers: one 128 x 4 atom of 512 bytes per 128 rows and 64 columns */
    EXPECT(nvfp4_sf_bytes(128, 64) == 512);
    EXPECT(nvfp4_sf_bytes(1, 16) == 512);
    EXPECT(nvfp4_sf_bytes(129, 128) == 4 * 512);
    EXPECT(nvfp4_sf_offset(0, 0, 64) == 0);
    EXPECT(nvfp4_sf_offset(1, 0, 64) == 16);
    EXPECT(nvfp4_sf_offset(32, 0, 64) == 4);
    EXPECT(nvfp4_sf_offset(0, 5, 512) == 512 + 1);
    EXPECT(nvfp4_sf_bytes_grouped(100, 64, 3) >= nvfp4_sf_bytes(100 + 3 * 127, 64));
    EXPECT(nvfp4_group_k_capacity(100, 3) == 320);
    EXPECT(nvfp4_quantize_2d_fused_workspace(5) == 32);

    /* argument checks come before any device work */
    nvfp4_tensor out;
    memset(&out, 0, sizeof out);
    EXPECT(nvfp4_quantize_1d(NULL, 16, 16, 16, NVFP4_ROUND_RNE, 0, NULL, &out, NULL) == NVFP4_ERR_NULL);
    static uint16_t x[16 * 17] __attribute__((aligned(16)));
    static uint8_t codes[16 * 8] __attribute__((aligned(16)));
    static uint8_t sf[512] __attribute__((aligned(16)));
    static float amax[1];
    out.codes = codes; out.sf = sf; out.amax = amax; out.rows = 16; out.cols = 16;
    EXPECT(nvfp4_quantize_1d(x, 16, 17, 17, NVFP4_ROUND_RNE, 0, NULL, &out, NULL) == NVFP4_ERR_SHAPE);
    EXPECT(nvfp4_quantize_1d(x + 1, 16, 16, 16, NVFP4_ROUND_RNE, 0, NULL, &out, NULL) == NVFP4_ERR_ALIGN);
    nvfp4_status s = nvfp4_quantize_1d(x, 16, 16, 16, NVFP4_ROUND_SR, 7, NULL, &out, NULL);
    EXPECT(s == NVFP4_ERR_DEVICE);

    /* the host-side injection hook reports its status without launching */
    nvfp4_debug_inject(NVFP4_ERR_TIMEOUT);
    EXPECT(nvfp4_quantize_1d(x, 16, 16, 16, NVFP4_ROUND_RNE, 0, NULL, &out, NULL) == NVFP4_ERR_TIMEOUT);
    nvfp4_debug_inject(NVFP4_OK);

    for (int st = NVFP4_OK; st <= NVFP4_ERR_LIMIT; ++st) {
        const char *m = nvfp4_status_string((nvfp4_status)st);
        EXPECT(m != NULL && strlen(m) > 0);
    }
    EXPECT(nvfp4_last_error() != NULL);
    printf("%s %d\n", fails ? "FAILED" : "OK", s);
    return fails != 0;
}
"""


def _need(tool):
    if shutil.which(tool) is None:
        pytest.skip(f"{tool} not installed")


def test_header_is_strict_c_and_cxx(tmp_path):
    _need("gcc")
    _need("g++")
    src = tmp_path / "h.c"
    src.write_text('#include "nvfp4.h"\nint main(void) { return (int)sizeof(nvfp4_tensor) == 0; }\n')
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{INC}", "-c",
                    str(src), "-o", str(tmp_path / "h.o")], check=True, capture_output=True)
    srcpp = tmp_path / "h.cpp"
    srcpp.write_text('#include "nvfp4.h"\nint main() { return sizeof(nvfp4_tensor) == 0; }\n')
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{INC}", "-c",
                    str(srcpp), "-o", str(tmp_path / "hpp.o")], check=True, capture_output=True)


def test_plain_c_program_against_the_library(tmp_path):
    _need("gcc")
    lib = os.path.join(PKG, "libnvfp4.so")
    if not os.path.exists(lib):
        from nvfp4_precision_02_b300 import build as nb
        nb.build()
    src = tmp_path / "consumer.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "consumer"
    r = subprocess.run(["gcc", "-std=gnu11", "-Wall", "-Wextra", "-Werror", f"-I{INC}", str(src), "-o", str(exe),
                        f"-L{PKG}", "-lnvfp4", f"-Wl,-rpath,{PKG}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # the program passes host buffers: it must never see a GPU, on any machine
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")



def test_c_example_compiles_and_links(tmp_path):
    """The C example (examples/fprop.c) compiles as C11 against the header
    and links against libnvfp4.so and the CUDA runtime (it is not run)."""
    _need("gcc")
    code = open(os.path.join(ROOT, "examples", "fprop.c")).read()
    assert "nvfp4_gemm(" in code
    src = tmp_path / "example.c"
    src.write_text(code + "\nint main(void) { return 0; }\n")
    cuda_inc, cuda_lib = "/usr/local/cuda/include", "/usr/local/cuda/lib64"
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("CUDA headers not installed")
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", f"-I{INC}", f"-I{cuda_inc}", str(src),
                        "-o", str(tmp_path / "example"), f"-L{PKG}", "-lnvfp4", f"-L{cuda_lib}", "-lcudart",
                        f"-Wl,-rpath,{PKG}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
