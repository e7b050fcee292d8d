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
              "spec_tree_verify_workspace", "spec_status_string", "spec_tree_attention_paged",
              "spec_kv_compact", "spec_kv_compact_paged", "spec_tree_verify_filtered",
              "spec_tree_verify_filtered_workspace", "spec_tree_build_workspace",
              "spec_tree_expand", "spec_tree_finalize", "spec_lm_head_stats",
              "spec_lm_head_stats_workspace", "spec_lm_head_pack", "spec_lm_head_stats_packed",
              "spec_tree_verify_greedy", "spec_tree_verify_head",
              "spec_tree_verify_head_workspace"):
        assert n in names


def test_binding_limits_match_the_header():
    from speculative_decoding_token_spec_gb300 import _binding
    text = open(HEADER).read()
    m = re.search(r"^#define\s+SPEC_NOALLOC_MAX_NODES\s+(\d+)", text, flags=re.M)
    assert m and _binding.NOALLOC_MAX_NODES == int(m.group(1))


def test_debug_wait_polls_setter(lib):
    assert lib.spec_debug_set_verify_wait_polls(0) == 0
    assert lib.spec_debug_set_verify_wait_polls(-1) == 0      # back to the default


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libspectree.so does not export {name}"


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, 1, 2, 4, 8, 16, 32, 64):
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


def test_paged_and_compaction_argument_errors(lib):
    """The new entry points reject bad arguments before any CUDA call (works without a GPU)."""
    fake = ctypes.c_void_p(256)
    null = None
    # paged attention: q, k_pages, v_pages, block_table, P, max_pages, num_pages, lens, parent,
    # out, lse, B, N, Hq, Hkv, D, scale, status, stream
    def attn(P=16, max_pages=8, num_pages=10, N=5, D=128, table=fake, scale=0.1):
        return lib.spec_tree_attention_paged(fake, fake, fake, table, P, max_pages, num_pages,
                                             fake, fake, fake, null, 1, N, 8, 8, D, scale, null,
                                             null)
    for P in (8, 24, 2048):            # page size: a power of two in [16, 1024]
        assert attn(P=P) == -2
    assert attn(table=null) == -1
    assert attn(max_pages=0) == -1
    assert attn(num_pages=0) == -1
    assert attn(D=96) == -2
    assert attn(N=65) == -1
    assert attn(P=16, max_pages=1, N=20) == -1        # Lmax = 16 < N
    assert attn(scale=float("nan")) == -1
    assert attn(P=1024, num_pages=1 << 20) == -2       # num_pages * Hkv * P >= 2^31
    # compaction: k, v, lens, accept_len, nodes, new_lens, B, N, Hkv, D, Lmax, status, stream
    lens = ctypes.c_void_p(512)
    def comp(new_lens=fake, k=fake, B=1, N=5, D=128, Lmax=100):
        return lib.spec_kv_compact(k, fake, lens, fake, fake, new_lens, B, N, 8, D, Lmax, null,
                                   null)
    assert comp(new_lens=lens) == -1                   # new lengths may not alias prefix_lens
    assert comp(k=null) == -1
    assert comp(N=65) == -1
    assert comp(D=80) == -2
    assert comp(B=0) == -1
    assert comp(Lmax=1 << 30, B=8) == -2               # B * Hkv * Lmax >= 2^31
    # paged compaction: k, v, table, P, max_pages, num_pages, lens, accept_len, nodes, new_lens,
    # B, N, Hkv, D, status, stream
    rc = lib.spec_kv_compact_paged(fake, fake, null, 16, 4, 4, lens, fake, fake, fake, 1, 5, 8,
                                   128, null, null)
    assert rc == -1
    rc = lib.spec_kv_compact_paged(fake, fake, fake, 0, 4, 4, lens, fake, fake, fake, 1, 5, 8,
                                   128, null, null)
    assert rc == -1


def test_filtered_verify_arguments(lib):
    """Filtered verification: workspace query and argument errors, all before any CUDA call."""
    base = lib.spec_tree_verify_workspace(2, 60, 32000)
    full = lib.spec_tree_verify_filtered_workspace(2, 60, 32000)
    assert full >= base + 2 * 60 * 32000 * 4 and full % 16 == 0
    assert lib.spec_tree_verify_filtered_workspace(1, 65, 100) == 0
    fake = ctypes.c_void_p(256)
    null = None

    def call(T=1.0, k=5, p=0.9, ws=1 << 30, probs=fake, N=5, V=1000):
        return lib.spec_tree_verify_filtered(fake, probs, fake, fake, fake, T, k, p, 1, N, V,
                                             fake, fake, fake, null, null, fake, ws, null, null)
    for k, p in ((-1, 0.9), (5, 0.0), (5, -0.2), (5, 1.5), (5, float("nan"))):
        assert call(k=k, p=p) == -1
    assert call(T=-1.0) == -1
    assert call(probs=null) == -1                    # T > 0 needs the draft distribution
    assert call(N=65) == -1
    need = lib.spec_tree_verify_filtered_workspace(1, 5, 1000)
    assert call(ws=need - 16) == -3                  # the filtered logits do not fit
    assert call(k=0, p=0.5, ws=need - 16) == -3      # top-p alone also filters


def test_tree_construction_arguments(lib):
    """Workspace query and argument errors of the tree construction, before any CUDA call."""
    assert lib.spec_tree_build_workspace(4, 10, 6) >= 4 * (128 + 16 * (1 + 10 + 5 * 100))
    assert lib.spec_tree_build_workspace(4, 17, 2) == 0       # K above SPEC_TREE_MAX_K
    assert lib.spec_tree_build_workspace(4, 16, 10) == 0      # pool above SPEC_TREE_MAX_POOL
    assert lib.spec_tree_build_workspace(0, 4, 2) == 0
    fake = ctypes.c_void_p(256)
    null = None
    ws = lib.spec_tree_build_workspace(2, 4, 3)

    def expand(V=100, K=4, D=3, level=1, logits=fake, nbytes=ws):
        return lib.spec_tree_expand(logits, 2, V, K, D, level, fake, nbytes, null, null, null,
                                    null)
    assert expand(logits=null) == -1
    assert expand(V=3) == -1                  # fewer tokens than K
    assert expand(level=0) == -1 and expand(level=4) == -1
    assert expand(K=0) == -1
    assert expand(nbytes=ws - 16) == -3

    def fin(N=10, K=4, D=3, nbytes=ws, out=fake):
        return lib.spec_tree_finalize(fake, nbytes, fake, 2, K, D, N, out, fake, null, null, null,
                                      null)
    assert fin(N=0) == -1 and fin(N=65) == -1
    assert fin(N=1 + 4 + 2 * 16 + 1) == -1    # more nodes than the construction can draft
    assert fin(out=null) == -1
    assert fin(nbytes=16) == -3


def test_lm_head_arguments(lib):
    """Workspace query and argument errors of the fused LM head, before any CUDA call."""
    assert lib.spec_lm_head_stats_workspace(60, 32000) == 250 * 60 * 16
    assert lib.spec_lm_head_stats_workspace(0, 10) == 0
    fake = ctypes.c_void_p(256)
    null = None
    ws = lib.spec_lm_head_stats_workspace(4, 1000)

    def call(M=4, H=64, V=1000, G=0, T=1.0, gi=null, og=null, nbytes=ws, h=fake):
        return lib.spec_lm_head_stats(h, fake, gi, M, H, V, G, T, fake, fake, fake, og, fake,
                                      nbytes, null, null)
    assert call(h=null) == -1
    assert call(H=60) == -1                 # H not a multiple of 8
    assert call(T=0.0) == -1 and call(T=float("nan")) == -1
    assert call(G=3) == -1                  # gathers without ids / outputs
    assert call(nbytes=ws - 16) == -3
    assert lib.spec_lm_head_packed_bytes(1000, 104) == 4 * 2 * 256 * 64 * 2  # padded tiles
    assert lib.spec_lm_head_packed_bytes(1000, 60) == 0
    assert lib.spec_lm_head_pack(fake, 1000, 64, fake, 16, null) == -3


def test_greedy_verify_arguments(lib):
    """Argument errors of the greedy verification, before any CUDA call."""
    fake = ctypes.c_void_p(256)
    null = None

    def call(B=2, N=10, V=100, am=fake, out=fake):
        return lib.spec_tree_verify_greedy(am, fake, fake, B, N, V, out, fake, fake, null, null,
                                           null)
    assert call(am=null) == -1 and call(out=null) == -1
    assert call(B=0) == -1 and call(N=0) == -1 and call(N=65) == -1 and call(V=0) == -1


def test_head_verify_arguments(lib):
    """Workspace query and argument errors of verification from the LM head, before any CUDA
    call."""
    assert lib.spec_tree_verify_head_workspace(1, 60, 4096, 32000, 6) > 0
    assert lib.spec_tree_verify_head_workspace(1, 60, 4096, 32000, 60) == 0  # depth >= N
    assert lib.spec_tree_verify_head_workspace(1, 60, 4100, 32000, 6) == 0   # H % 8
    assert lib.spec_tree_verify_head_workspace(1, 65, 4096, 32000, 6) == 0   # N > 64
    fake = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(260)
    null = None
    ws = lib.spec_tree_verify_head_workspace(2, 10, 64, 1000, 3)

    def call(B=2, N=10, H=64, V=1000, depth=3, T=1.0, h=fake, p=fake, nbytes=ws, wsp=fake,
             out=fake):
        return lib.spec_tree_verify_head(h, fake, 0, p, fake, fake, fake, T, B, N, H, V, depth,
                                         out, fake, fake, null, wsp, nbytes, null, null)
    assert call(h=null) == -1 and call(out=null) == -1
    assert call(h=odd) == -1 and call(p=odd) == -1      # 16-byte alignment
    assert call(p=null) == -1 and call(T=-1.0) == -1 and call(T=float("inf")) == -1
    assert call(H=60) == -1 and call(N=65) == -1 and call(B=0) == -1
    assert call(depth=10) == -1 and call(depth=-1) == -1
    assert call(nbytes=ws - 16) == -3 and call(wsp=null) == -3


def test_header_is_plain_c_and_a_c_program_links(lib, tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 (no CUDA or C++ types), and a C
    program built against it links to libspectree.so and calls it (entries that touch no GPU)."""
    import subprocess
    from speculative_decoding_token_spec_gb300 import _binding
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    so = _binding.lib_path()
    src = tmp_path / "use_spectree.c"
    src.write_text(
        '#include <stdio.h>\n#include "spectree.h"\n'
        "int main(void) {\n"
        "  printf(\"%s\\n\", spec_status_string(SPEC_ST_BAD_TREE));\n"
        "  return spec_tree_verify_workspace(1, 65, 10) == 0 ? 0 : 1;  /* N > 64: invalid */\n"
        "}\n")
    exe = tmp_path / "use_spectree"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.dirname(HEADER), str(src), "-o", str(exe), so,
                        "-Wl,-rpath," + os.path.dirname(so)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert run.returncode == 0, run.stderr
    assert "bad tree" in run.stdout
