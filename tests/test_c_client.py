"""The boundary from plain C (CPU): include/qgemv.h compiles on its own as C99 and
as C++17 with every warning an error, and a C99 program linked against the built
library packs matrices to the oracle's bytes without Python in the loop."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle as ORC
import workloads
import block_quantized_token_format_gb300 as qg
from _layout_ref import decode_device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
CLIENT = os.path.join(ROOT, "tests", "c", "abi_client.c")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None or shutil.which("g++") is None,
                                reason="needs gcc and g++")


def _compile(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.parametrize("lang", [["gcc", "-std=c99", "-x", "c"], ["g++", "-std=c++17", "-x", "c++"]])
def test_header_compiles_alone(lang, tmp_path):
    src = tmp_path / "inc.txt"
    src.write_text('#include "qgemv.h"\nint qg_header_probe(void) { return QG_OK + (int)QG_Q5_0; }\n')
    _compile(lang + ["-pedantic", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-c", str(src),
                     "-o", str(tmp_path / "inc.o")])


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    d = tmp_path_factory.mktemp("client")
    exe = d / "abi_client"
    lib_dir = os.path.dirname(qg._LIB_PATH)
    _compile(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-O1", "-I", INCLUDE, CLIENT,
              "-o", str(exe), "-L", lib_dir, "-lqgemv", "-Wl,-rpath," + lib_dir])
    return exe


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0", "affine4_g64", "bf16", "q5_0"])
@pytest.mark.parametrize("shape", [(5, 64), (9, 1088)])
def test_c_client_packs_to_oracle_bytes(client, fmt, shape, tmp_path):
    n_out, n_in = shape
    W = workloads.gaussian(321 + n_in, (n_out, n_in), 0.02)
    W[0] = 0.0
    W.astype(np.float32).tofile(tmp_path / "W.f32")
    canon_path, packed_path = tmp_path / "canon.bin", tmp_path / "packed.bin"
    r = subprocess.run([str(client), fmt, str(n_out), str(n_in), str(tmp_path / "W.f32"), str(canon_path),
                        str(packed_path)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    canon = np.fromfile(canon_path, dtype=np.uint8)
    packed = np.fromfile(packed_path, dtype=np.uint8)
    ref = ORC.quantize(fmt, W)
    assert np.array_equal(canon, ref)
    assert np.array_equal(decode_device(fmt, packed, n_out, n_in), ORC.dequantize(fmt, ref, n_out, n_in))


def test_c_client_refuses_an_unknown_format(client, tmp_path):
    r = subprocess.run([str(client), "q3_k", "1", "64", "W", "a", "b"], capture_output=True, text=True)
    assert r.returncode == 1 and "unknown format" in r.stderr
