"""The C-ABI library builds, loads and exports what include/*.h declares;
host-side argument checks answer without a GPU (CPU only)."""

import ctypes
import glob
import os
import re
import shutil

import pytest

from speculative_decoding_verification_73_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(spec_verify\w*)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not available")
    build.build()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "spec_verify" in declared and "spec_verify_init" in declared
    assert declared == set(binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_strerror_and_launch_count(lib):
    assert binding.strerror(0) == "success"
    for code in range(1, 9):
        assert binding.strerror(code) != "unknown error code"
    assert binding.strerror(99) == "unknown error code"
    assert binding.spec_verify_launches_per_call() == binding.SV_NUM_KERNELS == 2


def test_host_argument_checks_need_no_gpu(lib):
    ctx = ctypes.c_void_p()
    # every size check fails before any CUDA call is made
    bad = [(0, 4, 100, 1), (1, -1, 100, 1), (1, 256, 100, 1), (1, 4, 0, 1),
           (1, 4, (1 << 26) + 1, 1), (1, 4, 100, 2), ((1 << 20) + 1, 4, 100, 0)]
    for args in bad:
        assert lib.spec_verify_init(ctypes.byref(ctx), *args, None) == binding.SV_EINVAL
        assert ctx.value is None
    assert lib.spec_verify_init(None, 1, 1, 1, 0, None) == binding.SV_EINVAL
    # a null context is rejected by every entry point
    assert lib.spec_verify(None, 1, 1, 1, None, None, None, None, 0, None, None, None) == binding.SV_EINVAL
    assert lib.spec_verify_get_error(None, None) == binding.SV_EINVAL
    assert lib.spec_verify_debug_stats(None, 1, 1, None, None) == binding.SV_EINVAL
    assert lib.spec_verify_profile(None, 1) == binding.SV_EINVAL
    assert lib.spec_verify_profile_read(None, None, None) == binding.SV_EINVAL
    assert lib.spec_verify_destroy(None) == binding.SV_OK
    assert lib.spec_verify_debug_philox(0, None, None, -1, None) == binding.SV_EINVAL
    assert lib.spec_verify_debug_philox(0, None, None, 0, None) == binding.SV_OK
    assert lib.spec_verify_debug_seek_calls(None, 5) == binding.SV_EINVAL
    assert lib.spec_verify_debug_skip_row_stats(None, 1) == binding.SV_EINVAL
    assert lib.spec_verify_debug_late_cta(None, 1) == binding.SV_EINVAL
    assert lib.spec_verify_tree(None, 1, 1, 1, 0, None, None, None, None, None, 0, None, None, None,
                                None) == binding.SV_EINVAL
    assert lib.spec_verify_kv_commit(None, 0, 1, 1, 1, 1, 16, None, None, None, None, None, 0) \
        == binding.SV_EINVAL


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    """No CPU fallback: a missing library is a loud error."""
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load()
