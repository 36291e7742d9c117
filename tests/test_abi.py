"""The C-ABI library loads and exports every function include/tkv.h declares (no GPU needed:
nothing here launches work)."""
import ctypes
import os
import re
import subprocess

import pytest

from tiered_kv_cache_gqa_gb300 import EXPORTS, LIB_PATH, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tkv_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    if not os.path.exists(LIB_PATH):
        build.build()
    return LIB_PATH


def test_header_and_binding_agree():
    assert declared_functions() == sorted(EXPORTS)


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (tkv_\w+)", out))
    assert set(declared_functions()) <= exported


def test_status_strings_without_gpu(lib_path):
    import tiered_kv_cache_gqa_gb300 as tkv
    assert tkv.status_string(tkv.TKV_OK) == "ok"
    assert "poisoned" in tkv.status_string(tkv.TKV_ESTATE)


def test_create_rejects_bad_config_without_touching_a_gpu(lib_path):
    import tiered_kv_cache_gqa_gb300 as tkv
    lib = tkv.load()
    cfg = tkv.Config()
    cfg.num_layers, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim = 1, 6, 4, 64   # Hq % Hkv != 0
    cfg.batch, cfg.max_tokens = 1, 16
    cfg.ratio_t0 = 1.0
    ctx = ctypes.c_void_p()
    assert lib.tkv_create(ctypes.byref(cfg), ctypes.byref(ctx)) == tkv.TKV_EINVAL
    cfg.num_q_heads, cfg.head_dim = 4, 96                                               # head_dim
    assert lib.tkv_create(ctypes.byref(cfg), ctypes.byref(ctx)) == tkv.TKV_EINVAL
    cfg.head_dim, cfg.ratio_t0 = 64, 0.5                                                # ratios sum
    assert lib.tkv_create(ctypes.byref(cfg), ctypes.byref(ctx)) == tkv.TKV_EINVAL
    assert lib.tkv_append(None, 0, None, None, 1) == tkv.TKV_EINVAL


def header_struct_fields(name):
    """Field names, in order, of `typedef struct { ... } name;` in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\}\s*" + name + r"\s*;", text).group(1)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            names.append(re.match(r".*?\b(\w+)\s*(\[\w+\])?$", decl, flags=re.S).group(1))
    return names


@pytest.mark.parametrize("cname,pyname", [("tkv_config", "Config"), ("tkv_stats", "Stats"),
                                          ("tkv_prof_entry", "ProfEntry")])
def test_binding_structs_match_the_header(cname, pyname):
    import tiered_kv_cache_gqa_gb300 as tkv
    assert [f[0] for f in getattr(tkv, pyname)._fields_] == header_struct_fields(cname)


def test_host_link_probe_rejects_bad_sizes_without_a_gpu(lib_path):
    import tiered_kv_cache_gqa_gb300 as tkv
    assert tkv.tkv_measure_host_link(0, 1000)[0] == tkv.TKV_EINVAL          # below 1 MiB
    assert tkv.tkv_measure_host_link(0, (1 << 20) + 8)[0] == tkv.TKV_EINVAL  # not a multiple of 16
    assert tkv.tkv_measure_host_link(-1, 1 << 20)[0] == tkv.TKV_EINVAL


def test_noalloc_rejects_a_misaligned_cache_without_a_gpu(lib_path):
    """kv rows are copied in 16-byte units: a misaligned kv is refused before any CUDA call
    (the addresses are never dereferenced)."""
    import tiered_kv_cache_gqa_gb300 as tkv
    args = (1, 1, 8, 2, 128, 64)
    assert tkv.tkv_decode_dense_noalloc(0x10000, 0x20008, 0x30000, 0x40000, *args, stream=0) == tkv.TKV_EINVAL
    assert tkv.tkv_decode_dense_noalloc(0, 0x20000, 0x30000, 0x40000, *args, stream=0) == tkv.TKV_EINVAL
