"""Host-only checks of the C-ABI library: it loads, exports every entry point
declared in include/*.h, and rejects bad arguments without touching a GPU."""
import ctypes
import glob
import os
import re

import pytest

import protein_pair_representation_gate_b300 as pkg
from protein_pair_representation_gate_b300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(tri_attn_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    from protein_pair_representation_gate_b300 import build
    build.build()
    return pkg.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"tri_attn_create", "tri_attn_forward", "tri_attn_destroy"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert names >= set(pkg.EXPORTS)


def test_status_strings(lib):
    for s in range(7):
        assert pkg.status_string(s) and pkg.status_string(s) != "unknown status"
    assert pkg.status_string(99) == "unknown status"


def _cfg(**kw):
    base = dict(c_z=128, heads=4, head_dim=32, I_max=256, dtype=B.BF16, ln_eps=1e-5, key_chunks=1, force_simt=0)
    base.update(kw)
    return B.Config(**base)


@pytest.mark.parametrize("bad", [dict(c_z=0), dict(c_z=300), dict(heads=0), dict(head_dim=0), dict(head_dim=65),
                                 dict(heads=16, head_dim=32), dict(I_max=0), dict(I_max=20000), dict(dtype=7),
                                 dict(ln_eps=0.0), dict(ln_eps=float("nan")), dict(key_chunks=0), dict(key_chunks=65)])
def test_create_rejects_bad_config(lib, bad):
    h = ctypes.c_void_p(123)
    st = lib.tri_attn_create(ctypes.byref(_cfg(**bad)), ctypes.byref(h))
    assert st == B.EINVAL and h.value is None


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.tri_attn_create(None, ctypes.byref(h)) == B.EINVAL
    assert lib.tri_attn_create(ctypes.byref(_cfg()), None) == B.EINVAL
    w = B.Weights()
    assert lib.tri_attn_forward(None, 0, 8, 16, None, ctypes.byref(w), 256, 1 << 20, 4096, None) == B.EINVAL
    assert lib.tri_attn_workspace_bytes(None, 8) == 0
    assert lib.tri_attn_path(None) == -1
    assert lib.tri_attn_status_sync(None, None) == B.EINVAL
    assert lib.tri_attn_set_timing(None, 1) == B.EINVAL
    assert lib.tri_attn_kernel_times(None, None, None, 0) == -1
    assert lib.tri_attn_debug_inject(None, 1) == B.EINVAL
    lib.tri_attn_destroy(None)


def test_msa_entry_points_reject_null_arguments(lib):
    w = B.MsaWeights()
    assert lib.tri_attn_msa_workspace_bytes(None, 4, 8) == 0
    assert lib.tri_attn_msa_forward(None, 4, 8, 16, 256, None, 512, ctypes.byref(w), 0, 1024, 1 << 20, 4096,
                                    None) == B.EINVAL


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(FileNotFoundError):
        _load_missing(tmp_path)


def _load_missing(tmp_path):
    saved = B._lib
    B._lib = None
    try:
        B.load_library(str(tmp_path / "missing.so"))
    finally:
        B._lib = saved


def test_header_is_plain_c(tmp_path):
    """include/tri_attn.h compiles as C99 (no C++ in the ABI) and declares every
    exported entry point with a prototype a C caller can take the address of."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    names = sorted(declared_functions())
    src = tmp_path / "use_header.c"
    src.write_text('#include "tri_attn.h"\nvoid* entry_points[] = {\n' +
                   "".join(f"    (void*){n},\n" for n in names) + "};\n")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_no_cpu_fallback_without_a_gpu(lib):
    """Without a CUDA device the product path fails loudly: creating a context
    (triangle or MSA) raises instead of computing anything on the host."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    with pytest.raises(B.TriAttnError) as e:
        pkg.TriangleAttention(128, 4, 32, 64, "bf16")
    assert e.value.status in (B.ECUDA, B.EUNSUPPORTED)
    with pytest.raises(B.TriAttnError):
        pkg.MSARowAttention(128, 8, 32, 64, "bf16")
