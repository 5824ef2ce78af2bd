"""The C ABI loads, exports what include/ncp_attn.h declares, and rejects bad
arguments before touching the GPU (no compute call is made here)."""
import os
import re

import pytest

import non_causal_prefix_gb300 as ncp

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "ncp_attn.h")


@pytest.fixture(scope="module")
def lib():
    ncp.build(quiet=True)
    return ncp.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("attn_dense_fwd", "attn_prefix_fwd", "attn_status_string"):
        assert required in names
    assert set(names) == set(ncp.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for code in range(-7, 1):
        s = ncp.status_string(code)
        assert s and s != "unknown status"
    assert ncp.status_string(5) == "unknown status"


# Fake device addresses: validation fails before any CUDA call uses them.
A, B_, C, O = 0x10000000, 0x20000000, 0x30000000, 0x40000000


@pytest.mark.parametrize("args,want", [
    ((None, B_, C, O, 1, 128, 32, 64), ncp.ATTN_ERR_NULL),
    ((A, None, C, O, 1, 128, 32, 64), ncp.ATTN_ERR_NULL),
    ((A, B_, C, None, 1, 128, 32, 64), ncp.ATTN_ERR_NULL),
    ((A, B_, C, O, 0, 128, 32, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 0, 32, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 128, 0, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 128, 70000, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 128, 32, 96), ncp.ATTN_ERR_HEADDIM),
    ((A, B_, C, O, 1, 128, 32, 256), ncp.ATTN_ERR_HEADDIM),
    ((A, B_, C, O, 1, 128, 32, 0), ncp.ATTN_ERR_HEADDIM),
    ((A + 8, B_, C, O, 1, 128, 32, 64), ncp.ATTN_ERR_ALIGN),
    ((A, B_, C, O + 2, 1, 128, 32, 64), ncp.ATTN_ERR_ALIGN),
    ((A, B_, C, A, 1, 128, 32, 64), ncp.ATTN_ERR_ALIAS),
    ((A, B_, C, C + 16, 1, 128, 32, 64), ncp.ATTN_ERR_ALIAS),
    ((A, B_, C, A + 128 * 32 * 64 * 2 - 16, 1, 128, 32, 64), ncp.ATTN_ERR_ALIAS),
])
def test_dense_rejects(lib, args, want):
    assert lib.attn_dense_fwd(*args, None) == want


def test_dense_alias_boundary_is_exact(lib):
    # out starting exactly where q ends does not overlap q; it does overlap
    # nothing else here, so validation passes and the call would reach CUDA.
    # Check only the overlap arithmetic through a failing later argument.
    nbytes = 128 * 32 * 64 * 2
    assert lib.attn_dense_fwd(A, B_, C, A + nbytes, 1, 128, 32, 65, None) == ncp.ATTN_ERR_HEADDIM


@pytest.mark.parametrize("args,want", [
    ((A, None, None, B_, C, O, 1, 128, 1, 128, 32, 128), ncp.ATTN_ERR_NULL),
    ((A, B_, None, B_, C, O, 1, 128, 4, 128, 32, 128), ncp.ATTN_ERR_NULL),
    ((A, 0x50000000, 0x60000000, B_, C, O, 1, 128, -1, 128, 32, 128), ncp.ATTN_ERR_SHAPE),
    ((A, 0x50000000, 0x60000000, B_, C, O, 1, 128, 4, 0, 32, 128), ncp.ATTN_ERR_SHAPE),
    ((A, 0x50000000, 0x60000000, B_, C, O, 1, 0, 4, 128, 32, 128), ncp.ATTN_ERR_SHAPE),
    ((A, 0x50000000, 0x60000000, B_, C, O, 1, 128, 4, 128, 32, 80), ncp.ATTN_ERR_HEADDIM),
    ((A, 0x50000004, 0x60000000, B_, C, O, 1, 128, 4, 128, 32, 128), ncp.ATTN_ERR_ALIGN),
    ((A, 0x50000000, 0x60000000, B_, C, 0x50000000, 1, 128, 4, 128, 32, 128),
     ncp.ATTN_ERR_ALIAS),
])
def test_prefix_rejects(lib, args, want):
    assert lib.attn_prefix_fwd(*args, None) == want


# Fake image-id and key_valid addresses (16-byte aligned, apart from the tensors).
IDS, KV = 0x70000000, 0x78000000


@pytest.mark.parametrize("args,want", [
    ((A, B_, C, None, O, 1, 256, 32, 128), ncp.ATTN_ERR_NULL),
    ((A, None, C, IDS, O, 1, 256, 32, 128), ncp.ATTN_ERR_NULL),
    ((A, B_, C, IDS + 4, O, 1, 256, 32, 128), ncp.ATTN_ERR_ALIGN),
    ((A, B_, C, IDS, O, 1, 128 * 1024 + 1, 32, 128), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, IDS, O, 1, 0, 32, 128), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, IDS, O, 1, 256, 32, 96), ncp.ATTN_ERR_HEADDIM),
    # out over the id vector, and out over q
    ((A, B_, C, IDS, IDS - 256 * 32 * 128 * 2 + 16, 1, 256, 32, 128), ncp.ATTN_ERR_ALIAS),
    ((A, B_, C, IDS, A, 1, 256, 32, 128), ncp.ATTN_ERR_ALIAS),
])
def test_block_causal_rejects(lib, args, want):
    assert lib.attn_block_causal_fwd(*args, None) == want


@pytest.mark.parametrize("args,want", [
    ((A, None, C, O, 1, 128, 512, 32, 64), ncp.ATTN_ERR_NULL),
    ((A, B_, C, O, 1, 128, 0, 32, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 0, 512, 32, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 128, 512, 32, 32), ncp.ATTN_ERR_HEADDIM),
    ((A, B_ + 2, C, O, 1, 128, 512, 32, 64), ncp.ATTN_ERR_ALIGN),
    ((A, B_, C, B_ + 64, 1, 128, 512, 32, 64), ncp.ATTN_ERR_ALIAS),
])
def test_cross_rejects(lib, args, want):
    assert lib.attn_dense_cross_fwd(*args, None) == want


def masked(q=A, kc=B_, vc=C, kp=0x50000000, vp=0x60000000, ids=IDS, kv=KV, scale=0.1, out=O,
           B=1, Nq=256, Np=128, H=32, D=128):
    return (q, kc, vc, kp, vp, ids, kv, scale, out, B, Nq, Np, H, D)


@pytest.mark.parametrize("args,want", [
    (masked(ids=None), ncp.ATTN_ERR_NULL),
    (masked(kc=None), ncp.ATTN_ERR_NULL),
    (masked(kp=None), ncp.ATTN_ERR_NULL),      # a prefix needs its K and V
    (masked(ids=IDS + 8), ncp.ATTN_ERR_ALIGN),
    (masked(scale=0.0), ncp.ATTN_ERR_SHAPE),
    (masked(scale=-0.1), ncp.ATTN_ERR_SHAPE),
    (masked(scale=float("inf")), ncp.ATTN_ERR_SHAPE),
    (masked(scale=float("nan")), ncp.ATTN_ERR_SHAPE),
    (masked(Np=-1), ncp.ATTN_ERR_SHAPE),
    (masked(Nq=0), ncp.ATTN_ERR_SHAPE),
    (masked(Nq=128 * 1024, Np=1), ncp.ATTN_ERR_SHAPE),  # more positions than the tile table
    (masked(D=48), ncp.ATTN_ERR_HEADDIM),
    (masked(out=KV - 16), ncp.ATTN_ERR_ALIAS),  # out over key_valid
    (masked(out=IDS), ncp.ATTN_ERR_ALIAS),      # out over the ids
    (masked(out=0x50000000), ncp.ATTN_ERR_ALIAS),  # out over the prefix K
])
def test_masked_prefix_rejects(lib, args, want):
    assert lib.attn_masked_prefix_fwd(*args, None) == want


@pytest.mark.parametrize("args,want", [
    ((None, B_, C, O, 1, 128, 32, 64), ncp.ATTN_ERR_NULL),
    ((A, B_, C, O, 1, 128, 0, 64), ncp.ATTN_ERR_SHAPE),
    ((A, B_, C, O, 1, 128, 32, 100), ncp.ATTN_ERR_HEADDIM),
    ((A, B_, C + 4, O, 1, 128, 32, 64), ncp.ATTN_ERR_ALIGN),
    ((A, B_, C, C, 1, 128, 32, 64), ncp.ATTN_ERR_ALIAS),
])
def test_noalloc_rejects(lib, args, want):
    assert lib.attn_dense_fwd_noalloc(*args, None) == want


def test_debug_hook_rejects_unknown_mode(lib):
    assert lib.attn_debug_set_fault(7, 0) == ncp.ATTN_ERR_SHAPE
    assert lib.attn_debug_set_fault(0, 0) == ncp.ATTN_OK


def test_binding_raises_on_missing_library(monkeypatch, tmp_path):
    """The product path has no fallback: a missing library is an error."""
    from non_causal_prefix_gb300 import _binding, _build
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _binding.load_library()


def test_product_path_does_not_import_the_oracle():
    """Nothing in the package refers to the test-only oracle."""
    pkg = os.path.dirname(ncp.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
