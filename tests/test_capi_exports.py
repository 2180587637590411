"""The shared library loads and exports every function include/pagedkv.h declares,
and the binding declares exactly those.  CPU only: no compute call needs a GPU."""
import os
import re
import subprocess

import libbuild
from paged_kv_cache_146_gb300 import _native

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_parses():
    names = declared_functions()
    assert "paged_decode_attention" in names and "kv_cache_write" in names
    assert "kv_pool_create" in names and len(names) >= 20


def test_library_exports_every_declared_symbol():
    libbuild.ensure_built()
    out = subprocess.run(["nm", "-D", "--defined-only", _native.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_binding_covers_header():
    assert sorted(n for n, _, _ in _native.SIGNATURES) == declared_functions()
    lib = libbuild.ensure_built()
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_host_only_calls():
    lib = libbuild.ensure_built()
    assert lib.pkv_version() >= 10000
    assert lib.pkv_status_string(-2) == b"out of free blocks"
    assert lib.kv_bytes_per_token(40, 40, 128, 2) == 819200
    assert lib.kv_blocks_for_tokens(100, 16) == 7
    assert lib.kv_pool_bytes(64, 16, 2, 64, 0) == 64 * 2 * 16 * 64 * 2
    assert lib.paged_decode_workspace_bytes(4, 4, 2, 64, 8) > 0
    assert lib.paged_decode_workspace_bytes(4, 5, 2, 64, 8) == 0      # Hq not a multiple of Hkv
    # prefill: the staged size adds the fp16 copy of V ([S * maxb][Hkv][16][D] x 2 B)
    base = lib.paged_prefill_workspace_bytes(3, 500, 32, 8)
    staged = lib.paged_prefill_workspace_bytes_staged(3, 500, 32, 8, 128, 40)
    assert base > 0 and staged >= base + 3 * 40 * 8 * 16 * 128 * 2
    assert lib.paged_prefill_workspace_bytes_staged(3, 500, 32, 8, 96, 40) == 0   # head_dim
    assert lib.paged_prefill_workspace_bytes_staged(3, 500, 32, 8, 128, 0) == 0
