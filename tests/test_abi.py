"""CPU checks of the C ABI: the library loads, exports every function the
header declares, its structs match the ctypes mirrors byte for byte, and the
host-side validation rejects bad arguments before any launch (no GPU needed:
these calls fail before touching CUDA)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from long_context_sparse_21_b300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


def declared_functions():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^CSA_API [\w\s\*]+?\b((?:csa|hca)_\w+)\(", txt, flags=re.M)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 13
    lib = abi.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T ((?:csa|hca)_\w+)", out))
    assert set(names) <= exported


def test_struct_layouts_match_header():
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "csa.h"
#define P(T) printf(#T " %zu\n", sizeof(T));
#define O(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  P(csa_store) P(csa_cache_write_params) P(csa_compress_params) P(csa_index_params) P(csa_attend_params)
  O(csa_compress_params, dst) O(csa_compress_params, tail_gate) O(csa_index_params, keys)
  O(csa_index_params, score_capacity) O(csa_attend_params, kv) O(csa_attend_params, scale)
  O(csa_attend_params, lse) O(csa_cache_write_params, dst) O(csa_cache_write_params, status)
  O(csa_store, max_pages) O(csa_store, num_pages) O(csa_attend_params, flags) O(csa_index_params, flags)
  O(csa_attend_params, rope_base) O(csa_compress_params, rope_base) O(csa_compress_params, flags)
  O(csa_compress_params, bias_b) O(csa_compress_params, k_new_b) O(csa_compress_params, tail_gate_b)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "t.c"), os.path.join(d, "t")
        open(src, "w").write(prog)
        subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe])
        got = dict(l.rsplit(" ", 1) for l in subprocess.check_output([exe], text=True).splitlines())
    mirror = {"csa_store": abi.CStore, "csa_cache_write_params": abi.CCacheWriteParams,
              "csa_compress_params": abi.CCompressParams, "csa_index_params": abi.CIndexParams,
              "csa_attend_params": abi.CAttendParams}
    for name, cls in mirror.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
    for key, val in got.items():
        if "." in key:
            t, f = key.split(".")
            assert getattr(mirror[t], f).offset == int(val), key


def test_page_bytes_and_strings():
    assert abi.page_bytes(abi.FMT_KV_POOL_FP8, 2048) == 644 * 2048
    assert abi.page_bytes(abi.FMT_INDEX_POOL_BF16, 128) == 256 * 128
    assert abi.page_bytes(abi.FMT_INDEX_POOL_E2M1, 256) == 72 * 256
    assert abi.page_bytes(abi.FMT_KV_POOL_FP8, 100) == 0  # not a multiple of 128
    assert abi.lib().csa_abi_version() == abi.ABI_VERSION
    for s in range(8):
        assert abi.status_string(s)
    assert abi.status_string(99) == "unknown status"


def _store(fmt, dim, base, P=128, table=0x10000, max_pages=4, capacity=0, num_pages=16):
    return abi.CStore(fmt, dim, base, capacity, P, table, max_pages, num_pages)


def test_validation_rejects_before_launch():
    L = abi.lib()
    assert L.csa_compress(None, None) == abi.ERR_INVALID_ARG
    p = abi.CCompressParams()
    p.struct_size = 4  # too small
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_INVALID_ARG
    # misaligned pool base
    p = abi.CCompressParams(struct_size=ctypes.sizeof(abi.CCompressParams), mode=abi.COMPRESS_DENSE, batch=1, m=4,
                            dim=576, bias=0x100000, n_tokens=8, k=0x200000, k_dtype=abi.BF16, g=0x300000,
                            g_dtype=abi.F32, dst=_store(abi.FMT_KV_POOL_FP8, 576, 0x400010))
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_ALIGN
    # wrong entry width for the KV pool
    p.dim = 512
    p.dst = _store(abi.FMT_KV_POOL_FP8, 512, 0x400000)
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_UNSUPPORTED
    # page size not a multiple of 128
    p.dim = 576
    p.dst = _store(abi.FMT_KV_POOL_FP8, 576, 0x400000, P=100)
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_SHAPE
    # index: unsupported q dtype for the bf16 pool; workspace too small
    ip = abi.CIndexParams(struct_size=ctypes.sizeof(abi.CIndexParams), num_queries=2, batch=2, heads=64, dim=128,
                          m=4, max_pos=1000, q=0x100000, q_dtype=abi.F32, w=0x200000, pos=0x300000, idx=0x400000,
                          cnt=0x500000, top_k=64, score_dtype=abi.F32,
                          keys=_store(abi.FMT_INDEX_POOL_BF16, 128, 0x800000, max_pages=2))
    assert L.csa_index_topk(ctypes.byref(ip), None, 0, None) == abi.ERR_UNSUPPORTED
    ip.q_dtype = abi.BF16
    need = L.csa_index_topk_workspace_size(ctypes.byref(ip))
    assert need > 1024
    assert L.csa_index_topk(ctypes.byref(ip), 0x900000, need - 1, None) == abi.ERR_WORKSPACE
    assert L.csa_index_topk(ctypes.byref(ip), None, need, None) == abi.ERR_WORKSPACE
    # pool too small for the positions
    ip.max_pos = 10 ** 6
    assert L.csa_index_topk(ctypes.byref(ip), 0x900000, 1 << 30, None) == abi.ERR_SHAPE
    # attention: unsupported head count on the tensor-core path
    ap = abi.CAttendParams(struct_size=ctypes.sizeof(abi.CAttendParams), num_queries=1, batch=1, heads=32, dim=576,
                           m=4, max_pos=100, q=0x100000, q_dtype=abi.BF16, pos=0x200000, idx=0x300000,
                           cnt=0x400000, top_k=8, kv=_store(abi.FMT_KV_POOL_FP8, 576, 0x800000), window=128,
                           win=0x500000, win_dtype=abi.BF16, win_ring=128, scale=0.1, out=0x600000,
                           out_dtype=abi.BF16)
    assert L.csa_attend(ctypes.byref(ap), 0x900000, 1 << 20, None) == abi.ERR_UNSUPPORTED
    assert L.csa_attend_workspace_size(ctypes.byref(ap)) == 0
    # unknown flag bits
    ap.heads, ap.flags = 64, 4
    assert L.csa_attend(ctypes.byref(ap), 0x900000, 1 << 20, None) == abi.ERR_INVALID_ARG
    ap.flags = 0
    # a pool of no pages
    ap.kv = _store(abi.FMT_KV_POOL_FP8, 576, 0x800000, num_pages=0)
    assert L.csa_attend(ctypes.byref(ap), 0x900000, 1 << 20, None) == abi.ERR_SHAPE
    # the optional status word of the cache writer must be 4-byte aligned
    cw = abi.CCacheWriteParams(struct_size=ctypes.sizeof(abi.CCacheWriteParams), batch=1, n=4, first=0,
                               src=0x100000, dst=_store(abi.FMT_KV_POOL_FP8, 576, 0x800000), status=0x200002)
    assert L.csa_cache_write(ctypes.byref(cw), None) == abi.ERR_ALIGN
    assert L.csa_index_topk_noalloc_status(None, None) == abi.ERR_INVALID_ARG


def test_validation_limits_of_each_path():
    L = abi.lib()
    # append: the ring must hold a block; one cluster of 8 CTAs covers at most 640 dims
    p = abi.CCompressParams(struct_size=ctypes.sizeof(abi.CCompressParams), mode=abi.COMPRESS_APPEND, batch=2, m=4,
                            dim=576, bias=0x100000, seq_len=0x200000, k_new=0x300000, g_new=0x400000,
                            ring=0x500000, ring_size=2, tail_gate=0x600000,
                            dst=_store(abi.FMT_KV_POOL_FP8, 576, 0x800000))
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_SHAPE
    # overlapping compression: the b stream's bias is required; its append takes m <= 16
    p.ring_size, p.mode = 128, abi.COMPRESS_APPEND_AB
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_INVALID_ARG
    p.bias_b, p.m, p.ring_size = 0x700000, 32, 32
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_UNSUPPORTED
    p.m = 4
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_INVALID_ARG  # no b-stream tails
    p.k_new_b, p.g_new_b, p.tail_b, p.tail_gate_b = 0x710000, 0x720000, 0x730008, 0x740000
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_ALIGN
    p.mode, p.bias_b = abi.COMPRESS_APPEND, None
    p.ring_size, p.dim = 128, 704
    p.dst = _store(abi.FMT_DENSE_F32, 704, 0x800000, capacity=64)
    assert L.csa_compress(ctypes.byref(p), None) == abi.ERR_SHAPE
    # indexer: the tensor-core pools take 64 heads of 128 dims
    ip = abi.CIndexParams(struct_size=ctypes.sizeof(abi.CIndexParams), num_queries=2, batch=2, heads=32, dim=128,
                          m=4, max_pos=1000, q=0x100000, q_dtype=abi.BF16, w=0x200000, pos=0x300000, idx=0x400000,
                          cnt=0x500000, top_k=64, score_dtype=abi.BF16,
                          keys=_store(abi.FMT_INDEX_POOL_BF16, 128, 0x800000, max_pages=2))
    assert L.csa_index_topk(ctypes.byref(ip), 0x900000, 1 << 30, None) == abi.ERR_UNSUPPORTED
    assert L.csa_index_topk_workspace_size(ctypes.byref(ip)) == 0
    # attention: D = 576 on the FP8 pool, and a window source that is either an
    # exact ring of W rows or a raw sequence covering every position
    ap = abi.CAttendParams(struct_size=ctypes.sizeof(abi.CAttendParams), num_queries=1, batch=1, heads=64, dim=512,
                           m=4, max_pos=1000, q=0x100000, q_dtype=abi.BF16, pos=0x200000, idx=0x300000,
                           cnt=0x400000, top_k=8, kv=_store(abi.FMT_KV_POOL_FP8, 512, 0x800000, max_pages=4),
                           window=128, win=0x500000, win_dtype=abi.BF16, win_ring=128, scale=0.1, out=0x600000,
                           out_dtype=abi.BF16)
    assert L.csa_attend(ctypes.byref(ap), 0x900000, 1 << 20, None) == abi.ERR_UNSUPPORTED
    ap.dim = 576
    ap.kv = _store(abi.FMT_KV_POOL_FP8, 576, 0x800000, max_pages=4)
    ap.win_ring = 200  # neither W nor >= max_pos + 1
    assert L.csa_attend(ctypes.byref(ap), 0x900000, 1 << 20, None) == abi.ERR_UNSUPPORTED
    assert L.hca_attend_workspace_size(ctypes.byref(ap)) == 0


def test_binding_refuses_to_run_without_library(monkeypatch):
    monkeypatch.setattr(abi, "_lib", None)
    monkeypatch.setattr(abi, "LIB_PATH", "/nonexistent/libcsa.so")
    with pytest.raises(RuntimeError, match="libcsa.so not found"):
        abi.lib()
