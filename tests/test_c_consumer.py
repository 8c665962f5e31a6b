"""The ABI from plain C, without a GPU.

A C99 program compiled by gcc with -pedantic -Werror includes include/ttt.h, links
libttt_b300.so and makes the calls that need no device: status strings, workspace
sizes and argument errors. It also prints the size and field offsets of the option
and plan structs, which must match the ctypes mirrors in the Python binding, since
a caller from C and the binding hand the same bytes to the library.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import test_sequence_layers_06_b300 as ttt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include "ttt.h"

#define FIELD(T, f) printf(#T "." #f "=%zu\n", offsetof(T, f))

int main(void) {
  float dummy[4];
  ttt_plan plan;
  ttt_options opt = {0};
  printf("sizeof.ttt_options=%zu\n", sizeof(ttt_options));
  FIELD(ttt_options, wait_timeout_ns);
  FIELD(ttt_options, inject_stall);
  FIELD(ttt_options, force_path);
  FIELD(ttt_options, seg_len);
  FIELD(ttt_options, phase_events);
  FIELD(ttt_options, pieces);
  printf("sizeof.ttt_plan=%zu\n", sizeof(ttt_plan));
  FIELD(ttt_plan, path);
  FIELD(ttt_plan, seg_len);
  FIELD(ttt_plan, seg_count);
  FIELD(ttt_plan, kernels);
  FIELD(ttt_plan, affine);
  FIELD(ttt_plan, pieces);
  printf("str.ok=%s\n", ttt_status_str(TTT_OK));
  printf("str.timeout=%s\n", ttt_status_str(TTT_ERR_TIMEOUT));
  printf("ws.linear=%zu\n", ttt_workspace_bytes(2, 3, 100, 64, 16, TTT_VARIANT_LINEAR));
  printf("ws.mlp=%zu\n", ttt_workspace_bytes(2, 3, 100, 64, 16, TTT_VARIANT_MLP));
  printf("ws.bad=%zu\n", ttt_workspace_bytes(0, 3, 100, 64, 16, TTT_VARIANT_LINEAR));
  printf("ws.bwd=%zu\n", ttt_linear_bwd_workspace_bytes(2, 3, 100, 64, 16));
  printf("fwd.null=%d\n", (int)ttt_linear_fwd(NULL, NULL, NULL, TTT_BF16, NULL, NULL, 1, 1, 16, 64, 16,
                                              NULL, NULL, NULL, 0, NULL));
  printf("fwd.width=%d\n", (int)ttt_linear_fwd(dummy, dummy, dummy, TTT_F32, dummy, dummy, 1, 1, 16, 65, 16,
                                               dummy, dummy, dummy, 1u << 20, NULL));
  printf("plan.bad=%d\n", (int)ttt_linear_plan(1, 1, 16, 64, 0, TTT_BF16, &opt, &plan));
  printf("bwd.d65=%d\n", (int)ttt_linear_bwd(dummy, dummy, dummy, TTT_BF16, dummy, dummy, 1, 1, 16, 65, 16,
                                              dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 1u << 20,
                                              NULL));
  printf("ws.var_bias=%zu\n", ttt_linear_variant_workspace_bytes(TTT_INNER_BIAS, TTT_BF16, 2, 3, 40, 16, 16));
  printf("ws.var_ln=%zu\n", ttt_linear_variant_workspace_bytes(TTT_INNER_LN, TTT_BF16, 2, 3, 40, 16, 16));
  printf("ws.mlp_bwd=%zu\n", ttt_mlp_bwd_workspace_bytes(2, 3, 40, 16, 8));
  printf("mlp_bwd.d65=%d\n", (int)ttt_mlp_bwd(dummy, dummy, dummy, TTT_F32, dummy, dummy, dummy, 1, 1, 16, 65, 16,
                                              dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                              dummy, 1u << 20, NULL));
  printf("bias_ex.nows=%d\n", (int)ttt_linear_bias_fwd_ex(dummy, dummy, dummy, TTT_BF16, dummy, dummy, dummy, 1, 1,
                                                          16, 16, 16, dummy, dummy, dummy, NULL, 0, NULL));
  printf("ws.var_mom=%zu\n", ttt_linear_variant_workspace_bytes(TTT_INNER_MOMENTUM, TTT_BF16, 2, 3, 40, 64, 16));
  printf("ln_ex.nows=%d\n", (int)ttt_linear_ln_fwd_ex(dummy, dummy, dummy, TTT_BF16, dummy, dummy, dummy, dummy, 1,
                                                       1, 16, 64, 16, dummy, dummy, NULL, 0, NULL, &opt));
  printf("mom_ex.nows=%d\n", (int)ttt_linear_momentum_fwd_ex(dummy, dummy, dummy, TTT_BF16, dummy, dummy, dummy, 1,
                                                             1, 16, 64, 16, dummy, dummy, dummy, NULL, 0, NULL,
                                                             &opt));
  return 0;
}
"""


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is not installed")
    from test_sequence_layers_06_b300 import build
    build.build()
    lib_dir = os.path.dirname(ttt.LIB_PATH)
    work = tmp_path_factory.mktemp("c_consumer")
    src, exe = work / "consumer.c", work / "consumer"
    src.write_text(PROGRAM)
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", lib_dir, "-lttt_b300", f"-Wl,-rpath,{lib_dir}"],
                   check=True, capture_output=True, text=True)
    run = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120)
    return dict(line.split("=", 1) for line in run.stdout.splitlines())


def test_struct_layouts_match_the_binding(c_output):
    for name, mirror in (("ttt_options", ttt.ttt_options), ("ttt_plan", ttt.ttt_plan)):
        assert int(c_output[f"sizeof.{name}"]) == ctypes.sizeof(mirror), name
        for field, _ in mirror._fields_:
            assert int(c_output[f"{name}.{field}"]) == getattr(mirror, field).offset, (name, field)


def test_calls_from_c_agree_with_the_binding(c_output):
    lib = ttt.load_library()
    assert c_output["str.ok"] == lib.ttt_status_str(0).decode()
    assert c_output["str.timeout"] == lib.ttt_status_str(-4).decode()
    assert int(c_output["ws.linear"]) == ttt.ttt_workspace_bytes(2, 3, 100, 64, 16) >= 256
    assert int(c_output["ws.mlp"]) == ttt.ttt_workspace_bytes(2, 3, 100, 64, 16, variant=ttt.TTT_VARIANT_MLP) >= 256
    assert int(c_output["ws.bad"]) == 0
    assert int(c_output["ws.bwd"]) == ttt.ttt_linear_bwd_workspace_bytes(2, 3, 100, 64, 16) > 256


def test_variant_and_mlp_backward_calls_from_c(c_output):
    assert int(c_output["ws.var_bias"]) == ttt.ttt_linear_variant_workspace_bytes(
        ttt.TTT_INNER_BIAS, ttt.TTT_BF16, 2, 3, 40, 16, 16) > 256
    assert int(c_output["ws.var_ln"]) == 256
    assert int(c_output["ws.var_mom"]) == 256
    assert int(c_output["mom_ex.nows"]) == ttt.TTT_ERR_ARG
    assert int(c_output["ln_ex.nows"]) == ttt.TTT_ERR_ARG
    assert int(c_output["ws.mlp_bwd"]) == ttt.ttt_mlp_bwd_workspace_bytes(2, 3, 40, 16, 8) > 256
    assert int(c_output["mlp_bwd.d65"]) == -2   # d > 64
    assert int(c_output["bias_ex.nows"]) == -1  # no workspace


def test_argument_errors_from_c(c_output):
    assert int(c_output["fwd.null"]) == -1      # TTT_ERR_ARG: null pointers
    assert int(c_output["fwd.width"]) == -2     # TTT_ERR_UNSUPPORTED: d > 64
    assert int(c_output["plan.bad"]) == -1      # b < 1
    assert int(c_output["bwd.d65"]) == -2       # no backward kernel takes d > 64
