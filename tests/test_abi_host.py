"""Host-side checks of libtq that need no GPU: the library loads and exports
every entry point declared in include/tq.h, the host codebook builder and the
Householder QR agree with the oracle, and argument validation rejects bad
calls before touching the device."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

import kv_cache_vector_tq_gb300 as tq
from oracle import codebook as ocb
from oracle import rotation as orot
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "tq.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(tq.LIB_PATH):
        from kv_cache_vector_tq_gb300 import build
        build.build()
    return tq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(tq.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert tq.tq_version().startswith("tq ")
    assert L.tq_status_string(tq.TQ_ERR_TIMEOUT) == b"TQ_ERR_TIMEOUT"


@pytest.mark.parametrize("d,b,dens", [(128, 1, 0), (128, 2, 0), (128, 3, 0), (128, 4, 0),
                                      (128, 2, 1), (1536, 4, 0), (32, 3, 0)])
def test_host_codebook_matches_oracle(L, d, b, dens):
    cb = tq.tq_codebook_build(d, b, dens)
    ref = ocb.build_codebook(d, b, "beta" if dens == 0 else "gauss")
    K = 1 << b
    np.testing.assert_allclose(np.array(cb.centroid[:K]), ref["centroids"], rtol=0, atol=1e-9)
    np.testing.assert_allclose(np.array(cb.threshold[:K - 1]), ref["thresholds"], rtol=0, atol=1e-9)
    assert abs(cb.distortion - ref["distortion"]) < 1e-10
    # the fp32 thresholds the kernels use round identically
    np.testing.assert_array_equal(np.float32(cb.threshold[:K - 1]), np.float32(ref["thresholds"]))


@pytest.mark.parametrize("d", [2, 32, 128, 384])
def test_host_haar_rotation_matches_oracle(L, d):
    G = np.random.default_rng(d).standard_normal((d, d))
    Pi = tq.tq_rotation_haar(G)
    ref = orot.haar_rotation(G)
    assert np.abs(Pi - ref).max() < 1e-12 * max(1, d / 32)
    assert np.abs(Pi.T @ Pi - np.eye(d)).max() < 1e-13 * max(1, d / 32)


def test_codebook_validation(L):
    cb = tq.Codebook()
    assert L.tq_codebook_build(1, 2, 0, 0, 0, ctypes.byref(cb)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_codebook_build(128, 5, 0, 0, 0, ctypes.byref(cb)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_codebook_build(128, 2, 7, 0, 0, ctypes.byref(cb)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_codebook_build(128, 2, 0, 0, 0, None) == tq.TQ_ERR_INVALID_ARG


def test_ctx_validation_before_device(L):
    d = 128
    Pi = np.eye(d)
    out = ctypes.c_void_p()
    cb3 = tq.tq_codebook_build(d, 3)
    p = tq._ptr
    # Prod needs b >= 2, S, and a (b-1)-bit codebook
    assert L.tq_ctx_create(d, 1, tq.TQ_PROD, 0, p(Pi), p(Pi), ctypes.byref(cb3), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_ctx_create(d, 3, tq.TQ_PROD, 0, p(Pi), None, ctypes.byref(cb3), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_ctx_create(d, 3, tq.TQ_PROD, 0, p(Pi), p(Pi), ctypes.byref(cb3), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    # codebook dimension mismatch, bad d, bad bits
    cb64 = tq.tq_codebook_build(64, 3)
    assert L.tq_ctx_create(d, 3, tq.TQ_MSE, 0, p(Pi), None, ctypes.byref(cb64), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_ctx_create(100, 3, tq.TQ_MSE, 0, p(Pi), None, ctypes.byref(cb3), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_ctx_create(d, 5, tq.TQ_MSE, 0, p(Pi), None, ctypes.byref(cb3), ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    # Hadamard order not 2^k or 12·2^k; signs must be ±1
    cb160 = tq.tq_codebook_build(160, 3)
    s160 = np.ones(160)
    assert L.tq_ctx_create(160, 3, tq.TQ_MSE, 1, p(s160), None, ctypes.byref(cb160), ctypes.byref(out)) == tq.TQ_ERR_UNSUPPORTED
    assert not out.value
    assert L.tq_ctx_destroy(None) == tq.TQ_ERR_INVALID_ARG


def test_mixed_ctx_validation_before_device(L):
    """b + 1/2 bits: two codebooks (b and b + 1 bits), b = 1..3, d = 128 (either
    rotation: a Hadamard context passes validation and fails only for want of
    a device here)."""
    p = tq._ptr
    out = ctypes.c_void_p()

    def pair(d, b0, b1):
        arr = (tq.Codebook * 2)()
        arr[0], arr[1] = tq.tq_codebook_build(d, b0), tq.tq_codebook_build(d, b1)
        return ctypes.cast(arr, ctypes.POINTER(tq.Codebook)), arr

    cb, keep = pair(128, 2, 3)
    bad, keep2 = pair(128, 2, 4)  # second codebook not b + 1 bits
    cb4, keep3 = pair(128, 4, 4)
    cb256, keep4 = pair(256, 2, 3)
    I128, I256 = np.eye(128), np.eye(256)
    assert L.tq_ctx_create(128, 2, tq.TQ_MIXED, 0, p(I128), None, bad, ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_ctx_create(128, 4, tq.TQ_MIXED, 0, p(I128), None, cb4, ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_ctx_create(256, 2, tq.TQ_MIXED, 0, p(I256), None, cb256, ctypes.byref(out)) == tq.TQ_ERR_UNSUPPORTED
    st = L.tq_ctx_create(128, 2, tq.TQ_MIXED, 1, p(np.ones(128)), None, cb, ctypes.byref(out))
    assert st not in (tq.TQ_ERR_INVALID_ARG, tq.TQ_ERR_UNSUPPORTED)
    if st == tq.TQ_OK:
        assert L.tq_ctx_destroy(out) == tq.TQ_OK
        out = ctypes.c_void_p()
    assert L.tq_ctx_create(128, 2, 3, 0, p(I128), None, cb, ctypes.byref(out)) == tq.TQ_ERR_INVALID_ARG
    assert not out.value


def test_unpack_validation(L):
    c = tq.Codes()
    assert L.tq_unpack_indices(ctypes.byref(c), 0, 1, None, None) == tq.TQ_ERR_INVALID_ARG


def test_words_per_vector_rule():
    # 16-byte padding of the packed stream, as the oracle's canonical packing
    from oracle.quantizer import words_per_vector
    assert [words_per_vector(128, b) for b in (1, 2, 3, 4)] == [4, 8, 12, 16]
    assert words_per_vector(32, 3) == 4 and words_per_vector(3072, 4) == 384
    assert math.ceil(4 * 1536 / 32) == 192


def test_per_device_cache_logic(tmp_path):
    """Kernel attributes, SM counts and occupancy answers are kept per device
    (tq_once.h): compile the header's host test with g++ and run it."""
    import shutil
    import subprocess
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    exe = tmp_path / "per_device_value_test"
    src = os.path.join(ROOT, "tests", "native", "per_device_value_test.cpp")
    inc = os.path.join(ROOT, "kv_cache_vector_tq_gb300", "csrc")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", inc, src, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
