"""The library's host code under AddressSanitizer and UndefinedBehaviorSanitizer
(CPU only; compute-sanitizer is not available for the device code, whose
checks are the parity tests on small shapes and the kernels' own bounds).

The library is rebuilt with -fsanitize=address,undefined on its host code
into a temporary directory, then a separate Python process loads it with the
sanitizer runtimes preloaded and runs every host path that needs no GPU:
argument checks of each entry point, a sweep of invalid layer configurations
(every field out of range, extreme integers, NaN and infinite epsilons),
every status string, the allocation-free projection's checks, and a valid
configuration whose creation fails at its first CUDA call on a machine
without a GPU (the weights are re-tiled on the host and everything is
released on the error path).  Any sanitizer report fails the test."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SAN_FLAGS = []
for _f in ("-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=undefined",
           "-fno-omit-frame-pointer"):
    SAN_FLAGS += ["-Xcompiler", _f]

CHECKS = r'''
import ctypes, math, sys
sys.path.insert(0, ROOT)
import numpy as np
from gated_deltanet_hybrid_gb300 import abi
from gated_deltanet_hybrid_gb300.inputs import TINY, make_weights

lib = abi.load_library(LIB)
E = abi.DN_EINVAL

# NULL and range checks of every entry point
assert lib.dn_create(None, None, None, None) == E
assert lib.dn_step(None, 1, None, None, None, None, 1, None) == E
assert lib.dn_set_state(None, 0, 1, None, None, None, 0) == E
assert lib.dn_get_state(None, 0, 1, None, None, None, 0) == E
assert lib.dn_stack_step(None, 1, 1, None, None, None, 1e-6, None) == E
assert lib.dn_debug_fail_next(None, -5) == E
assert lib.dn_debug_expire_wait(None, 1000) == E
assert lib.dn_profile_next_step(None, None) == E
assert lib.dn_step_kernels(None, 1) == 0
lib.dn_destroy(None)
for code in (0, -1, -2, -3, -4, -5, 7, -2**31, 2**31 - 1):
    assert len(lib.dn_strerror(code)) > 0

# invalid configurations: one field at a time, extreme values included
base = dict(hidden=256, qk=2, v=4, dk=32, dv=32, conv_k=4, max_batch=2, l2=1e-6, ne=1e-6, qs=1.0, fl=0)
bad = {"hidden": [0, 8, 250, 16400, -16, 2**31 - 1, -2**31],
       "qk": [0, -1, 3, 2**31 - 1, -2**31], "v": [0, 65, -4, 2**31 - 1, -2**31],
       "dk": [0, 16, 48, 512, -32, 2**31 - 1], "dv": [0, 16, 96, 512, -2**31],
       "fl": [2, 3, -1, 2**31 - 1],
       "conv_k": [0, 1, 9, -4, 2**31 - 1], "max_batch": [0, 1025, -1, 2**31 - 1, -2**31],
       "l2": [0.0, -1e-6, math.nan, -math.inf], "ne": [0.0, -1.0, math.nan],
       "qs": [math.nan]}
h = ctypes.c_void_p()
w = abi.dn_weights()
n = 0
for field, values in bad.items():
    for val in values:
        c = dict(base, **{field: val})
        cfg = abi.dn_config(c["hidden"], c["qk"], c["v"], c["dk"], c["dv"], c["conv_k"], c["max_batch"],
                            c["l2"], c["ne"], c["qs"], c["fl"])
        assert lib.dn_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h)) == E, (field, val)
        assert h.value is None
        n += 1
# a valid configuration with a missing weight array
cfg = abi.dn_config(256, 2, 4, 32, 32, 4, 2, 1e-6, 1e-6, 1.0)
assert lib.dn_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h)) == E

# the allocation-free projection's host checks
p16 = ctypes.c_void_p(16 * 1024)  # 16-byte aligned, never dereferenced: the checks fail first
for M, K, B in ((0, 64, 1), (64, 8, 1), (64, 72, 1), (64, 64, 0), (64, 64, 9), (20000, 64, 1)):
    assert lib.dn_proj_i8_noalloc(p16, p16, p16, p16, M, K, B, None) == E, (M, K, B)
assert lib.dn_proj_i8_noalloc(None, p16, p16, p16, 64, 64, 1, None) == E
assert lib.dn_proj_i8_noalloc(ctypes.c_void_p(16 * 1024 + 4), p16, p16, p16, 64, 64, 1, None) == E

# a valid layer: weights re-tiled on the host, then the first CUDA call fails
# (no GPU here) and everything is released
wts = make_weights(TINY, np.random.default_rng(0))
rc = abi.dn_create(TINY, wts, 2, stream=0, check=False)
assert rc == abi.DN_ECUDA or rc == abi.DN_ENOMEM, rc
assert lib.dn_device_bytes() == 0
print("host paths ok", n)
'''


def _runtime(name: str) -> str | None:
    gcc = shutil.which("gcc")
    if gcc is None:
        return None
    p = subprocess.run([gcc, f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


@pytest.fixture(scope="module")
def sanitized_lib(tmp_path_factory):
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc sanitizer runtimes not installed")
    from gated_deltanet_hybrid_gb300 import build as b
    d = tmp_path_factory.mktemp("san")
    lib = b.build(extra=SAN_FLAGS, lib=str(d / "libdn_san.so"), build_dir=str(d / "obj"))
    return lib, f"{asan} {ubsan}"


def test_host_paths_under_asan_and_ubsan(sanitized_lib):
    lib, preload = sanitized_lib
    env = dict(os.environ, LD_PRELOAD=preload, CUDA_VISIBLE_DEVICES="",
               ASAN_OPTIONS="detect_leaks=0:verify_asan_link_order=0:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    code = f"ROOT = {ROOT!r}\nLIB = {lib!r}\n" + CHECKS
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    report = r.stdout[-2000:] + r.stderr[-4000:]
    assert r.returncode == 0, report
    assert "host paths ok" in r.stdout, report
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, report
