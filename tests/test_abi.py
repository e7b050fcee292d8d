"""C-ABI checks that need no GPU: the library builds, loads, exports every symbol the header
declares, and rejects bad arguments synchronously without touching a device."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spectree.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="CUDA toolkit not available")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?[\s\*]+(spec_\w+)\s*\(",
                                 text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_token_spec_gb300 import _binding, build
    build.build()
    return _binding.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("spec_tree_attention", "spec_tree_verify", "spec_tree_attention_workspace",
              "spec_tree_verify_workspace", "spec_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libspectree.so does not export {name}"


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, 1, 2, 4, 8, 16):
        assert lib.spec_status_string(code)
    assert b"unknown" in lib.spec_status_string(12345)


def test_verify_workspace_query(lib):
    assert lib.spec_tree_verify_workspace(2, 60, 32000) >= 2 * 60 * 32
    assert lib.spec_tree_verify_workspace(1, 65, 100) == 0
    assert lib.spec_tree_verify_workspace(0, 5, 100) == 0


def test_argument_errors_are_synchronous(lib):
    """Bad scalars / NULL pointers are rejected before any CUDA call (works without a GPU)."""
    fake = ctypes.c_void_p(256)
    null = None
    # verify: NULL logits
    rc = lib.spec_tree_verify(null, fake, fake, fake, fake, 1.0, 1, 5, 10, fake, fake, fake,
                              null, null, fake, 1 << 20, null, null)
    assert rc == -1
    # verify: negative and NaN temperature
    for T in (-0.5, float("nan"), float("inf")):
        rc = lib.spec_tree_verify(fake, fake, fake, fake, fake, T, 1, 5, 10, fake, fake, fake,
                                  null, null, fake, 1 << 20, null, null)
        assert rc == -1
    # verify: T > 0 requires draft probabilities
    rc = lib.spec_tree_verify(fake, null, fake, fake, fake, 1.0, 1, 5, 10, fake, fake, fake,
                              null, null, fake, 1 << 20, null, null)
    assert rc == -1
    # verify: N out of range
    for N in (0, 65):
        rc = lib.spec_tree_verify(fake, fake, fake, fake, fake, 1.0, 1, N, 10, fake, fake, fake,
                                  null, null, fake, 1 << 20, null, null)
        assert rc == -1
    # verify: workspace too small
    rc = lib.spec_tree_verify(fake, fake, fake, fake, fake, 1.0, 1, 5, 10, fake, fake, fake,
                              null, null, fake, 8, null, null)
    assert rc == -3
    # attention: unsupported head dim, bad GQA grouping, NULL output
    args = [fake] * 5
    rc = lib.spec_tree_attention(*args, fake, null, 1, 5, 8, 8, 96, 200, 0.1, fake, 1 << 20,
                                 null, null)
    assert rc == -2
    rc = lib.spec_tree_attention(*args, fake, null, 1, 5, 8, 3, 128, 200, 0.1, fake, 1 << 20,
                                 null, null)
    assert rc == -1
    rc = lib.spec_tree_attention(*args, null, null, 1, 5, 8, 8, 128, 200, 0.1, fake, 1 << 20,
                                 null, null)
    assert rc == -1
    rc = lib.spec_tree_attention(*args, fake, null, 1, 65, 8, 8, 128, 200, 0.1, fake, 1 << 20,
                                 null, null)
    assert rc == -1
    rc = lib.spec_tree_attention(*args, fake, null, 1, 5, 8, 8, 128, 4, 0.1, fake, 1 << 20,
                                 null, null)
    assert rc == -1   # Lmax < N
    for scale in (0.0, -0.1, float("nan")):   # the softmax scale must be positive and finite
        rc = lib.spec_tree_attention(*args, fake, null, 1, 5, 8, 8, 128, 200, scale, fake,
                                     1 << 20, null, null)
        assert rc == -1
