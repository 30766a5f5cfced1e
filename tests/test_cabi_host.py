"""The C-ABI library on the host (no GPU needed): it loads, exports every
symbol include/kvq.h declares, and rejects bad arguments before launching
anything."""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(kvq.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return kvq.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(10):
        assert kvq.status_string(s) != "unknown status"
    assert "FP16" in kvq.status_string(kvq.KVQ_ERR_RANGE)
    assert kvq.status_string(99) == "unknown status"


def _cache(**kw):
    c = kvq.CacheStruct()
    c.batch, c.heads, c.head_dim, c.bits, c.group = 1, 2, 128, 2, 32
    c.chunk_tokens, c.n_chunks, c.len, c.head_slot = 10, 3, 0, 0
    # fake, aligned, never dereferenced: every call below fails validation
    # (or is a no-op) before anything touches device memory
    c.k_codes = c.v_codes = c.k_sz = c.v_sz = 0x10000
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_cache_bytes(lib):
    c = _cache()
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.kvq_cache_bytes(ctypes.byref(c), ctypes.byref(cb), ctypes.byref(sb)) == 0
    assert cb.value == 2 * 30 * 32 and sb.value == 2 * 30 * 4 * 4
    c = _cache(bits=4, group=64)
    assert lib.kvq_cache_bytes(ctypes.byref(c), ctypes.byref(cb), ctypes.byref(sb)) == 0
    assert cb.value == 2 * 30 * 64 and sb.value == 2 * 30 * 2 * 4
    kb, vb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.kvq_cache_meta_bytes(ctypes.byref(c), ctypes.byref(kb), ctypes.byref(vb)) == 0
    assert kb.value == vb.value == sb.value


def test_cache_bytes_per_channel_keys(lib):
    """Per-channel keys: k_sz holds d (step, zero) words per 128-token block
    of every chunk slot (blocks restart at each slot); v_sz is unchanged;
    kvq_cache_bytes reports the larger of the two."""
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    kb, vb = ctypes.c_size_t(), ctypes.c_size_t()
    for chunk, n_chunks in ((10, 3), (300, 4), (4680, 4)):
        c = _cache(key_mode=kvq.KEYS_PER_CHANNEL, chunk_tokens=chunk, n_chunks=n_chunks)
        assert lib.kvq_cache_meta_bytes(ctypes.byref(c), ctypes.byref(kb), ctypes.byref(vb)) == 0
        bpc = -(-chunk // 128)
        assert kb.value == 2 * n_chunks * bpc * 128 * 4
        assert vb.value == 2 * chunk * n_chunks * 4 * 4
        assert lib.kvq_cache_bytes(ctypes.byref(c), ctypes.byref(cb), ctypes.byref(sb)) == 0
        assert sb.value == max(kb.value, vb.value)
        assert cb.value == 2 * chunk * n_chunks * 32


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, kvq.KVQ_ERR_UNSUPPORTED),
    ("bits", 3, kvq.KVQ_ERR_UNSUPPORTED),
    ("group", 16, kvq.KVQ_ERR_UNSUPPORTED),
    ("batch", 0, kvq.KVQ_ERR_INVALID_ARG),
    ("n_chunks", 0, kvq.KVQ_ERR_INVALID_ARG),
    ("len", 31, kvq.KVQ_ERR_INVALID_ARG),
    ("head_slot", 3, kvq.KVQ_ERR_INVALID_ARG),
    ("key_mode", 2, kvq.KVQ_ERR_INVALID_ARG),
    ("key_mode", -1, kvq.KVQ_ERR_INVALID_ARG),
])
def test_bad_geometry(lib, field, value, status):
    c = _cache(**{field: value})
    assert lib.kvq_cache_bytes(ctypes.byref(c), None, None) == status
    assert lib.kvq_quantize_append(ctypes.byref(c), 0x10000, 0x10000, 5, None) == status


def test_append_window_rules_match_oracle(lib):
    """Every refused append is refused on the host, with the state untouched;
    the accepted ones agree with the oracle's ring rules."""
    C, n = 10, 3
    cases = [(20, 2, 4), (24, 0, 10), (30, 1, 9), (0, 0, 11), (10, 0, 10), (5, 0, 10)]
    for length, head, n_new in cases:
        want = O.ring_append(length, head, n_new, C, n)
        c = _cache(len=length, head_slot=head)
        if want is None:
            st = lib.kvq_quantize_append(ctypes.byref(c), 0x10000, 0x10000, n_new, None)
            assert st == kvq.KVQ_ERR_CAPACITY, (length, head, n_new, st)
            assert (c.len, c.head_slot) == (length, head)
    # zero-length append is a no-op that succeeds without touching anything
    c = _cache(len=24, head_slot=0)
    assert lib.kvq_quantize_append(ctypes.byref(c), 0x10000, 0x10000, 0, None) == 0
    assert (c.len, c.head_slot) == (24, 0)


def test_append_argument_checks(lib):
    c = _cache()
    assert lib.kvq_quantize_append(ctypes.byref(c), 0, 0x10000, 5, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_quantize_append(ctypes.byref(c), 0x10008, 0x10000, 5, None) == kvq.KVQ_ERR_ALIGNMENT
    assert lib.kvq_quantize_append(ctypes.byref(c), 0x10000, 0x10000, -1, None) == kvq.KVQ_ERR_INVALID_ARG
    c = _cache(k_codes=0x10004)
    assert lib.kvq_quantize_append(ctypes.byref(c), 0x10000, 0x10000, 5, None) == kvq.KVQ_ERR_ALIGNMENT
    assert lib.kvq_quantize_append(None, 0x10000, 0x10000, 5, None) == kvq.KVQ_ERR_INVALID_ARG


def test_attention_argument_checks(lib):
    c = _cache(len=30)
    ws = lib.kvq_workspace_bytes(ctypes.byref(c), 100, 10)
    assert ws >= 2 * (2 * 100 * 128 * 2) + 2 * 10 * 128 * 2
    f = lib.kvq_attention_corrected
    P = 0x10000
    # bad correction mode, bad flags, bad scale, missing output, workspace too small
    assert f(ctypes.byref(c), P, P, P, 100, 10, 0.1, 7, 0, P, ws, P, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, 0.1, 3, 0, P, ws, P, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, 0.1, 1, 16, P, ws, P, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, float("nan"), 1, 0, P, ws, P, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, -1.0, 1, 0, P, ws, P, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, 0.1, 1, 0, P, ws, None, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, 0.1, 1, 0, P, ws - 16, P, None, None, None) == 1
    assert f(ctypes.byref(c), P, P, P, 100, 10, 0.1, 1, 0, P, ws, P, P, None, None) == 1
    assert f(ctypes.byref(c), P + 2, P, P, 100, 10, 0.1, 1, 0, P, ws, P, None, None, None) == 6
    # nothing to attend to
    c0 = _cache(len=0)
    assert f(ctypes.byref(c0), P, P, P, 100, 0, 0.1, 1, 0, P, ws, P, None, None, None) == 1
    # no queries: a no-op
    assert f(ctypes.byref(c), P, P, P, 0, 10, 0.1, 1, 1, P, ws, P, None, None, None) == 0
    g = lib.kvq_attention_mass
    assert g(ctypes.byref(c), P, P, 100, 10, 0.1, 1, 0, P, ws, None, None, None) == 1


def test_rotate_argument_checks(lib):
    sb = (ctypes.c_uint32 * 4)(0, 0, 0, 0)
    assert lib.kvq_rotate(0x10000, 4, 96, sb, 0x10000, None, None) == kvq.KVQ_ERR_UNSUPPORTED
    assert lib.kvq_rotate(0x10000, 4, 64, sb, 0x10000, 0x10000, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_rotate(0x10000, 4, 64, sb, None, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_rotate(0x10000, 0, 64, sb, 0x10000, None, None) == 0
    assert lib.kvq_set_wait_limit_ns(0) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_selftest_wait_timeout(0, None) == kvq.KVQ_ERR_INVALID_ARG


def test_sign_bits_roundtrip():
    rng = np.random.default_rng(0)
    s = np.where(rng.integers(0, 2, 128) == 1, -1.0, 1.0)
    words = kvq.sign_bits(s)
    back = [(-1.0 if (words[c >> 5] >> (c & 31)) & 1 else 1.0) for c in range(128)]
    assert np.array_equal(back, s)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    """The allocation-free entry point refuses, on the host, problems whose
    scratch would not fit its built-in buffer."""
    c = _cache(len=30, heads=64)
    P = 0x10000
    n = 4096   # 64 heads x 4096 rows x 128 x 2 B x 2 (hi, lo) > 32 MiB
    assert lib.kvq_workspace_bytes(ctypes.byref(c), n, n) > kvq.NOALLOC_SCRATCH_BYTES
    st = lib.kvq_attention_corrected_noalloc(ctypes.byref(c), P, P, P, n, n, 0.1, 1, 0, P, None,
                                             None, None)
    assert st == kvq.KVQ_ERR_TOO_LARGE
    assert "scratch" in kvq.status_string(st)


def _unsplit_scratch(bh, n_q, n_r, d, kch_tiles=0):
    """Bytes of the unsplit launch's scratch as kvq.h defines it: the rotated
    query as FP16 high and low parts and the rotated current values (each
    region rounded up to 256 bytes), the per-channel key table, and two
    floats per (batch, head) for the per-head kernel choice."""
    up = lambda x: -(-x // 256) * 256
    return (2 * up(bh * n_q * d * 2) + up(bh * n_r * d * 2) + up(kch_tiles * bh * n_q * 4)
            + 2 * up(bh * 4))


def test_noalloc_refusal_is_the_unsplit_scratch_of_the_current_window(lib):
    """The allocation-free entry point refuses a problem exactly when the
    unsplit launch's scratch exceeds its buffer, not when
    kvq_workspace_bytes (sized for the split of a full window) does: just
    below the bound the call passes the size check (and, with no GPU here,
    fails at its first CUDA call instead); just above it is refused."""
    P = 0x10000
    c = _cache(len=30, heads=64)
    bh, d, n_r = 64, 128, 16
    # largest n_q whose unsplit scratch fits the 32 MiB buffer
    n_q = max(n for n in range(1000, 1200) if _unsplit_scratch(bh, n, n_r, d) <= kvq.NOALLOC_SCRATCH_BYTES)
    assert _unsplit_scratch(bh, n_q + 1, n_r, d) > kvq.NOALLOC_SCRATCH_BYTES
    args = lambda n: (ctypes.byref(c), P, P, P, n, n_r, 0.1, 1, 0, P, None, None, None)
    assert lib.kvq_attention_corrected_noalloc(*args(n_q)) != kvq.KVQ_ERR_TOO_LARGE
    assert lib.kvq_attention_corrected_noalloc(*args(n_q + 1)) == kvq.KVQ_ERR_TOO_LARGE
    # per-channel keys: the table of the cached key blocks of the current
    # window counts too (30 tokens in 3 slots of 10: one block each)
    ch = _cache(len=30, heads=64, key_mode=kvq.KEYS_PER_CHANNEL)
    n_q = max(n for n in range(900, 1200)
              if _unsplit_scratch(bh, n, n_r, d, 3) <= kvq.NOALLOC_SCRATCH_BYTES)
    argc = lambda n: (ctypes.byref(ch), P, P, P, n, n_r, 0.1, 1, 0, P, None, None, None)
    assert lib.kvq_attention_corrected_noalloc(*argc(n_q)) != kvq.KVQ_ERR_TOO_LARGE
    assert lib.kvq_attention_corrected_noalloc(*argc(n_q + 1)) == kvq.KVQ_ERR_TOO_LARGE


def test_binding_makes_the_tensors_device_current():
    """The library launches on the current device and looks its status word
    up there: the binding switches to the tensors' device for each call and
    refuses a stream of another device (checked without running a kernel)."""
    import torch
    assert isinstance(kvq._on_device(torch.device("cpu")), type(__import__("contextlib").nullcontext()))
    assert isinstance(kvq._on_device(None), type(__import__("contextlib").nullcontext()))
    g = kvq._on_device(torch.device("cuda", 1))
    assert isinstance(g, torch.cuda.device) and g.idx == 1

    class FakeStream:
        device = torch.device("cuda", 1)
        cuda_stream = 1234

    with pytest.raises(ValueError, match="stream belongs to cuda:1"):
        kvq._stream(FakeStream(), torch.device("cuda", 0))
    assert kvq._stream(FakeStream(), torch.device("cuda", 1)).value == 1234


def test_workspace_bytes_per_channel_keys(lib):
    """Per-channel keys add one fp32 per query row and cached key block (the
    blocks of every chunk slot: n_chunks x ceil(chunk / 128)) to the
    workspace, rounded to 256 bytes; nothing else changes."""
    for chunk, n_chunks, n_q, n_r in ((300, 4, 100, 10), (4680, 4, 4680, 4680), (1, 3, 7, 1)):
        tok = _cache(chunk_tokens=chunk, n_chunks=n_chunks)
        ch = _cache(chunk_tokens=chunk, n_chunks=n_chunks, key_mode=kvq.KEYS_PER_CHANNEL)
        w_tok = lib.kvq_workspace_bytes(ctypes.byref(tok), n_q, n_r)
        w_ch = lib.kvq_workspace_bytes(ctypes.byref(ch), n_q, n_r)
        tiles = n_chunks * -(-chunk // 128)
        table = -(-(tiles * 2 * n_q * 4) // 256) * 256          # 2 = batch x heads of _cache
        assert w_ch - w_tok == table, (chunk, n_chunks, w_ch, w_tok, table)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_caller():
    """include/kvq.h is a C header: a C11 program compiles against it, links
    libkvq.so and gets the same sizes and host-side errors."""
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    pkg = os.path.join(root, "quantized_kv_cache_quantize_gb300")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "c_abi_check")
        subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                               "-o", exe, os.path.join(here, "c_abi_check.c"), "-L", pkg, "-lkvq",
                               "-Wl,-rpath," + pkg])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("ok")


def test_binding_checks_shapes_before_passing_pointers(lib):
    """The library cannot see the size of a device buffer, so the binding
    checks every tensor against the cache's batch, heads and head_dim before
    it passes the pointer on; on the host (CPU tensors) a tensor of the right
    shape gets as far as the device check, one of the wrong shape stops at
    the shape check, and nothing reaches the library."""
    import torch
    cache = kvq.KVCache(1, 2, 128, 2, 32, 10, 3, np.ones(128), device="cpu")
    bf = dict(dtype=torch.bfloat16)
    good = torch.zeros(1, 2, 4, 128, **bf)
    for bad in (torch.zeros(1, 3, 4, 128, **bf), torch.zeros(2, 2, 4, 128, **bf),
                torch.zeros(1, 2, 4, 64, **bf), torch.zeros(2, 4, 128, **bf)):
        with pytest.raises(ValueError, match="shape"):
            kvq.quantize_append(cache, bad, bad)
        with pytest.raises(ValueError, match="shape"):
            kvq.attention_corrected(cache, bad, good, good)
        with pytest.raises(ValueError, match="shape"):
            kvq.attention_corrected(cache, good, bad, bad)
        with pytest.raises(ValueError, match="shape"):
            kvq.attention_corrected_noalloc(cache, bad, good, good)
        with pytest.raises(ValueError, match="shape"):
            kvq.attention_mass(cache, bad, good)
    with pytest.raises(ValueError, match="v_cur"):
        kvq.attention_corrected(cache, good, good, torch.zeros(1, 2, 5, 128, **bf))
    with pytest.raises(ValueError, match="k_new and v_new"):
        kvq.quantize_append(cache, good, torch.zeros(1, 2, 5, 128, **bf))
    # right shapes: stopped by the dtype / device check instead
    for call in (lambda: kvq.quantize_append(cache, good, good),
                 lambda: kvq.attention_corrected(cache, good, good, good),
                 lambda: kvq.attention_corrected_noalloc(cache, good, good, good),
                 lambda: kvq.attention_mass(cache, good, good)):
        with pytest.raises(ValueError, match="CUDA bfloat16"):
            call()
    assert cache.len == 0 and cache.head_slot == 0
    with pytest.raises(ValueError, match="shape of q"):
        kvq._check_out(good, torch.zeros(1, 2, 5, 128, **bf))
    with pytest.raises(ValueError, match="CUDA bfloat16"):
        kvq._check_out(good, torch.zeros(1, 2, 4, 128, **bf))
    # the workspace size passed on is in bytes, whatever the element type
    assert kvq._workspace_arg(torch.zeros(6, dtype=torch.float32), torch.device("cpu"))[1] == 24
    with pytest.raises(ValueError, match="workspace"):
        kvq._workspace_arg(torch.zeros(4, 4, dtype=torch.uint8).t(), torch.device("cpu"))


def test_binding_mirrors_the_header():
    """The Python binding's constants and its ctypes copy of kvq_cache agree
    with include/kvq.h: enum values and #defines parsed from the header, and
    every field's offset and the struct's size from a C compiler."""
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    consts = dict((k, int(v)) for k, v in re.findall(r"\b(KVQ_[A-Z0-9_]+)\s*=\s*(\d+)", src))
    consts.update((k, int(v)) for k, v in re.findall(r"#define\s+(KVQ_[A-Z0-9_]+)\s+(\d+)", src))
    py = {"KVQ_CORR_NONE": kvq.CORR_NONE, "KVQ_CORR_TAYLOR": kvq.CORR_TAYLOR,
          "KVQ_CORR_EXACT": kvq.CORR_EXACT, "KVQ_FLAG_PRECISE_QUERY": kvq.FLAG_PRECISE_QUERY,
          "KVQ_FLAG_NO_KV_SPLIT": kvq.FLAG_NO_KV_SPLIT, "KVQ_FLAG_ONE_CTA": kvq.FLAG_ONE_CTA,
          "KVQ_FLAG_STAGED_WORDS": kvq.FLAG_STAGED_WORDS,
          "KVQ_KEYS_PER_TOKEN": kvq.KEYS_PER_TOKEN, "KVQ_KEYS_PER_CHANNEL": kvq.KEYS_PER_CHANNEL,
          "KVQ_KEY_BLOCK": kvq.KEY_BLOCK}
    py.update((k, getattr(kvq, k)) for k in consts if k.startswith(("KVQ_OK", "KVQ_ERR_")))
    assert set(py) == set(consts), set(py) ^ set(consts)
    for k, v in consts.items():
        assert py[k] == v, (k, py[k], v)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("needs a C compiler")
    fields = [f[0] for f in kvq.CacheStruct._fields_]
    prog = ["#include <stddef.h>", "#include <stdio.h>", '#include "kvq.h"', "int main(void) {",
            '  printf("%zu\\n", sizeof(kvq_cache));']
    prog += [f'  printf("%zu\\n", offsetof(kvq_cache, {f}));' for f in fields]
    prog += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as tmp:
        c_path, exe = os.path.join(tmp, "layout.c"), os.path.join(tmp, "layout")
        with open(c_path, "w") as f:
            f.write("\n".join(prog) + "\n")
        subprocess.check_call([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", exe, c_path])
        got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(kvq.CacheStruct)
    for name, off in zip(fields, got[1:]):
        assert getattr(kvq.CacheStruct, name).offset == off, name
