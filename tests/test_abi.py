"""CPU checks of the C ABI: the library builds, loads without a GPU, exports every symbol the
header declares, and refuses bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import invariant_hybrid_attention_gb300 as g4
from invariant_hybrid_attention_gb300 import build as g4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    g4build.build()
    return g4.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "g4attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(g4attn_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("g4attn_prefill", "g4attn_decode", "g4attn_rope_apply"):
        assert n in names
    assert set(names) == set(g4.EXPORTS)


def declaration_blocks():
    """(comment, declared function names) for each comment of the header after the file comment:
    the functions declared between that comment and the next one."""
    text = open(os.path.join(ROOT, "include", "g4attn.h")).read()
    parts = re.split(r"(/\*.*?\*/)", text, flags=re.S)
    blocks, comment = [], None
    for part in parts[2:]:          # parts[1] is the file comment
        if part.startswith("/*"):
            comment = part
        else:
            names = re.findall(r"\b(g4attn_\w+)\s*\(", part)
            if names:
                blocks.append((comment or "", names))
    return blocks


def test_every_entry_point_cites_its_passage():
    """Each declared call sits under a comment that names the passage of the pages it implements
    (an RFC section and row or rule), or says that the pages have no counterpart of it."""
    seen = set()
    for comment, names in declaration_blocks():
        flat = " ".join(re.sub(r"\n\s*\*(?!/)", " ", comment).split())
        assert re.search(r"RFC section \d", flat) or "no counterpart" in flat, names
        seen.update(names)
    assert seen == set(declared_functions())


def test_provenance_names_the_exponential(lib):
    """The softmax exponential's flavour is a declared choice, so the provenance record names it."""
    for layer in (g4.sliding_layer(), g4.global_layer()):
        buf = ctypes.create_string_buffer(2048)
        n = lib.g4attn_provenance(ctypes.byref(layer), buf, len(buf))
        assert n > 0
        rec = buf.value.decode()
        assert "exp=ex2.approx.ftz.f32" in rec and "fallback=none" in rec and "accumulator=fp32" in rec


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    syms = os.popen(f"nm -D {g4.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\sT\s{name}$", syms, flags=re.M), name


def test_status_strings(lib):
    for s in range(7):
        assert len(g4.status_string(s)) > 0
    assert g4.status_string(g4.G4_ERR_UNSUPPORTED) == "unsupported geometry"


def test_unsupported_geometry_fails_closed(lib):
    bad = g4.sliding_layer()
    bad.head_dim = 128
    assert lib.g4attn_provenance(ctypes.byref(bad), None, 0) == -1
    cache = g4.g4attn_cache(16, 32, None, 4, 16)
    st = lib.g4attn_prefill(ctypes.byref(bad), 16, 16, 16, 8, 16, 16, 16, 1, ctypes.byref(cache), 16, 1, 16, None)
    assert st == g4.G4_ERR_UNSUPPORTED
    glob = g4.global_layer()
    glob.rope_partial = 0.5
    assert lib.g4attn_rope_apply(ctypes.byref(glob), 16, 16, 4, 1, 16, None) == g4.G4_ERR_UNSUPPORTED
    win = g4.global_layer()
    win.window = 1024          # a window on a global layer is not a supported geometry
    assert lib.g4attn_decode_workspace_bytes(ctypes.byref(win), 4, 4) == 0
    s = g4.sliding_layer()
    s.window = 0
    assert lib.g4attn_rope_apply(ctypes.byref(s), 16, 16, 4, 1, 16, None) == g4.G4_ERR_UNSUPPORTED


def test_invalid_arguments_refused_on_host(lib):
    s = g4.sliding_layer()
    cache = g4.g4attn_cache(16, 32, None, 4, 16)
    # NULL q
    assert lib.g4attn_prefill(ctypes.byref(s), None, 16, 16, 8, 16, 16, 16, 1, ctypes.byref(cache), 16, 1, 16,
                              None) == g4.G4_ERR_INVALID
    # misaligned q
    assert lib.g4attn_prefill(ctypes.byref(s), 18, 16, 16, 8, 16, 16, 16, 1, ctypes.byref(cache), 16, 1, 16,
                              None) == g4.G4_ERR_INVALID
    # B = 0
    assert lib.g4attn_prefill(ctypes.byref(s), 16, 16, 16, 8, 16, 16, 16, 0, ctypes.byref(cache), 16, 1, 16,
                              None) == g4.G4_ERR_INVALID
    # page size other than 16
    c8 = g4.g4attn_cache(16, 32, None, 4, 8)
    assert lib.g4attn_prefill(ctypes.byref(s), 16, 16, 16, 8, 16, 16, 16, 1, ctypes.byref(c8), 16, 1, 16,
                              None) == g4.G4_ERR_UNSUPPORTED
    # a global layer given a V tensor (K==V takes none), or without its rotated-column pages
    gl = g4.global_layer()
    cg = g4.g4attn_cache(16, 32, 48, 4, 16)
    assert lib.g4attn_prefill(ctypes.byref(gl), 16, 16, None, 8, 16, 16, 16, 1,
                              ctypes.byref(g4.g4attn_cache(16, None, None, 4, 16)), 16, 1, 16,
                              None) == g4.G4_ERR_INVALID
    assert lib.g4attn_prefill(ctypes.byref(gl), 16, 16, 16, 8, 16, 16, 16, 1, ctypes.byref(cg), 16, 1, 16,
                              None) == g4.G4_ERR_INVALID
    # scale must be finite and positive
    s2 = g4.sliding_layer(softmax_scale=-1.0)
    assert lib.g4attn_rope_apply(ctypes.byref(s2), 16, 16, 4, 1, 16, None) == g4.G4_ERR_INVALID
    # too small a decode workspace
    ws_need = lib.g4attn_decode_workspace_bytes(ctypes.byref(s), 4, 100)
    assert ws_need > 0
    assert lib.g4attn_decode(ctypes.byref(s), 16, 16, 16, 16, 4, ctypes.byref(cache), 16, 100, 16, 16,
                             ws_need - 1, None) == g4.G4_ERR_INVALID


def test_norm_arguments_refused_on_host(lib):
    s, gl = g4.sliding_layer(), g4.global_layer()
    cs = g4.g4attn_cache(16, 32, None, 4, 16)
    cg = g4.g4attn_cache(16, None, 48, 4, 16)

    def pre(layer, cache, norms, v):
        return lib.g4attn_prefill_normed(ctypes.byref(layer), ctypes.byref(norms) if norms else None, 16, 16, v, 8,
                                         16, 16, 16, 1, ctypes.byref(cache), 16, 1, 16, None)
    for eps in (0.0, -1e-6, float("inf"), float("nan")):   # eps must be finite and positive
        assert pre(s, cs, g4.g4attn_norms(16, 16, 1, eps), 16) == g4.G4_ERR_INVALID
    assert pre(s, cs, g4.g4attn_norms(18, None, 0, 1e-6), 16) == g4.G4_ERR_INVALID    # misaligned weight
    assert pre(s, cs, g4.g4attn_norms(None, 18, 0, 1e-6), 16) == g4.G4_ERR_INVALID
    assert pre(s, cs, g4.g4attn_norms(None, None, 2, 1e-6), 16) == g4.G4_ERR_INVALID  # v_norm is 0 or 1
    # K==V: the key norm and the unit value norm come together
    assert pre(gl, cg, g4.g4attn_norms(None, 16, 0, 1e-6), None) == g4.G4_ERR_UNSUPPORTED
    assert pre(gl, cg, g4.g4attn_norms(16, None, 1, 1e-6), None) == g4.G4_ERR_UNSUPPORTED
    assert lib.g4attn_kv_append_normed(ctypes.byref(gl), ctypes.byref(g4.g4attn_norms(None, 16, 0, 1e-6)), 16, None,
                                       8, 16, 16, 16, 1, ctypes.byref(cg), 16, 1, None) == g4.G4_ERR_UNSUPPORTED
    assert lib.g4attn_decode_normed(ctypes.byref(gl), ctypes.byref(g4.g4attn_norms(None, None, 1, 1e-6)), 16, 16,
                                    None, 16, 4, ctypes.byref(cg), 16, 100, 16, 16, 1 << 30,
                                    None) == g4.G4_ERR_UNSUPPORTED



def test_misaligned_image_span_refused_on_host(lib):
    """g4attn_prefill_vision reads spans as int32 pairs: a pointer off an 8-byte boundary is
    refused before anything runs (the other pointers here are fake and never touched)."""
    s, gl = g4.sliding_layer(), g4.global_layer()
    cs = g4.g4attn_cache(16, 32, None, 4, 16)
    cg = g4.g4attn_cache(16, None, 48, 4, 16)
    for layer, cache, v in ((s, cs, 16), (gl, cg, None)):
        assert lib.g4attn_prefill_vision(ctypes.byref(layer), None, 16, 16, v, 8, 16, 16, 16, 1, 20,
                                         ctypes.byref(cache), 16, 1, 16, None) == g4.G4_ERR_INVALID

def test_decode_exact_workspace_refused_on_host(lib):
    """The exact decode's rows live in the caller's workspace: too small or misaligned is refused
    before any launch (the other pointers are fake and never touched)."""
    s = g4.sliding_layer()
    cs = g4.g4attn_cache(16, 32, None, 4, 16)
    need = lib.g4attn_decode_exact_workspace_bytes(5)
    assert need >= 5 * 4 * 4 and need % 16 == 0
    assert lib.g4attn_decode_exact_workspace_bytes(0) == 0
    assert lib.g4attn_decode_exact(ctypes.byref(s), None, 16, 16, 16, 16, 5, ctypes.byref(cs), 16, 1, 16, 16,
                                   need - 16, None) == g4.G4_ERR_INVALID
    assert lib.g4attn_decode_exact(ctypes.byref(s), None, 16, 16, 16, 16, 5, ctypes.byref(cs), 16, 1, 16, 24,
                                   need, None) == g4.G4_ERR_INVALID


def test_split_steps_append_and_new_calls_refused_on_host(lib):
    """The split prefill steps, the plain append, the exact decode and the vision prefill refuse
    bad arguments before any launch (the other pointers are fake and never touched)."""
    s, gl = g4.sliding_layer(), g4.global_layer()
    bad = g4.sliding_layer()
    bad.n_q_heads = 16
    cs = g4.g4attn_cache(16, 32, None, 4, 16)
    cg = g4.g4attn_cache(16, None, 48, 4, 16)
    L = ctypes.byref
    # g4attn_prefill_stage: misaligned out; unsupported geometry
    assert lib.g4attn_prefill_stage(L(s), 16, 16, 16, 8, 16, 16, 16, 1, L(cs), 16, 1, 24, None) == g4.G4_ERR_INVALID
    assert lib.g4attn_prefill_stage(L(bad), 16, 16, 16, 8, 16, 16, 16, 1, L(cs), 16, 1, 16, None) == \
        g4.G4_ERR_UNSUPPORTED
    # g4attn_prefill_attend: NULL q_start; B = 0; unsupported geometry; misaligned raw queries
    assert lib.g4attn_prefill_attend(L(s), None, 8, None, 16, 16, 1, L(cs), 16, 1, 16, None) == g4.G4_ERR_INVALID
    assert lib.g4attn_prefill_attend(L(s), None, 8, 16, 16, 16, 0, L(cs), 16, 1, 16, None) == g4.G4_ERR_INVALID
    assert lib.g4attn_prefill_attend(L(bad), None, 8, 16, 16, 16, 1, L(cs), 16, 1, 16, None) == \
        g4.G4_ERR_UNSUPPORTED
    # raw queries off a 16-byte boundary
    assert lib.g4attn_prefill_attend(L(s), 24, 8, 16, 16, 16, 1, L(cs), 16, 1, 16, None) == g4.G4_ERR_INVALID
    # g4attn_kv_append: a V tensor on a K==V layer; no V on a sliding layer; negative T
    assert lib.g4attn_kv_append(L(gl), 16, 16, 8, 16, 16, 16, 1, L(cg), 16, 1, None) == g4.G4_ERR_INVALID
    assert lib.g4attn_kv_append(L(s), 16, None, 8, 16, 16, 16, 1, L(cs), 16, 1, None) == g4.G4_ERR_INVALID
    assert lib.g4attn_kv_append(L(s), 16, 16, -1, 16, 16, 16, 1, L(cs), 16, 1, None) == g4.G4_ERR_INVALID
    # g4attn_decode_exact: unsupported geometry; B = 0; NULL seq_len
    need = lib.g4attn_decode_exact_workspace_bytes(4)
    assert lib.g4attn_decode_exact(L(bad), None, 16, 16, 16, 16, 4, L(cs), 16, 1, 16, 16, need, None) == \
        g4.G4_ERR_UNSUPPORTED
    assert lib.g4attn_decode_exact(L(s), None, 16, 16, 16, 16, 0, L(cs), 16, 1, 16, 16, need, None) == \
        g4.G4_ERR_INVALID
    assert lib.g4attn_decode_exact(L(s), None, 16, 16, 16, None, 4, L(cs), 16, 1, 16, 16, need, None) == \
        g4.G4_ERR_INVALID
    # g4attn_prefill_vision: unsupported geometry (the span itself aligned)
    assert lib.g4attn_prefill_vision(L(bad), None, 16, 16, 16, 8, 16, 16, 16, 1, 16, L(cs), 16, 1, 16, None) == \
        g4.G4_ERR_UNSUPPORTED


def test_workspace_sizes(lib):
    s, gl = g4.sliding_layer(), g4.global_layer()
    # sliding: a 1024-key window touches at most 5 chunks of 256 keys; partial = (m, l) + 256 floats
    n = lib.g4attn_decode_workspace_bytes(ctypes.byref(s), 64, 2048)
    assert n >= 64 * 32 * 5 * (256 + 2) * 4
    # global: 32768 keys = 32 chunks of 1024
    n = lib.g4attn_decode_workspace_bytes(ctypes.byref(gl), 64, 2048)
    assert n >= 64 * 32 * 32 * (512 + 2) * 4
    # a page table longer than the 262144-position limit needs no more chunks (and no int overflow)
    at_limit = lib.g4attn_decode_workspace_bytes(ctypes.byref(gl), 2, 262144 // 16)
    assert at_limit >= 2 * 32 * 256 * (512 + 2) * 4
    assert lib.g4attn_decode_workspace_bytes(ctypes.byref(gl), 2, 2**31 - 1) == at_limit
    assert lib.g4attn_decode_workspace_bytes(ctypes.byref(s), 2, 2**31 - 1) == \
        lib.g4attn_decode_workspace_bytes(ctypes.byref(s), 2, 2048)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(g4, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        g4.load(str(tmp_path / "nope.so"))


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "invariant_hybrid_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "oracle/" not in text and "oracle." not in text, f


def test_decode_static_scratch_limit(lib):
    """The static-scratch decode refuses, on the host and before any CUDA call, a step whose
    workspace would exceed the static buffer; the documented examples sit at the boundary."""
    hdr = open(os.path.join(ROOT, "include", "g4attn.h")).read()
    assert "#define G4ATTN_DECODE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)" in hdr
    cap = g4.DECODE_STATIC_SCRATCH_BYTES
    s, gl = g4.sliding_layer(1024), g4.global_layer()
    ws = lambda layer, B, mp: lib.g4attn_decode_workspace_bytes(ctypes.byref(layer), B, mp)
    assert ws(s, 203, 2048) <= cap < ws(s, 204, 2048)
    assert ws(gl, 15, 2048) <= cap < ws(gl, 16, 2048)
    cache = g4.g4attn_cache(16, None, 16, 4, 16)
    st = lib.g4attn_decode_static(ctypes.byref(gl), 16, 16, None, 16, 16, ctypes.byref(cache), 16, 2048, 16, None)
    assert st == g4.G4_ERR_SCRATCH
    assert "static scratch" in g4.status_string(g4.G4_ERR_SCRATCH)
    assert lib.g4attn_decode_static(ctypes.byref(gl), 16, 16, None, 16, 0, ctypes.byref(cache), 16, 2048, 16,
                                    None) == g4.G4_ERR_INVALID
    bad = g4.global_layer()
    bad.head_dim = 256
    assert lib.g4attn_decode_static(ctypes.byref(bad), 16, 16, None, 16, 1, ctypes.byref(cache), 16, 8, 16,
                                    None) == g4.G4_ERR_UNSUPPORTED


def test_wait_limit_is_set_and_read_on_the_host(lib):
    """The kernels' wait bound is a host setting read at each launch: 0 .. 2e9 ns, 2 s by default;
    larger values are refused and leave it unchanged. No CUDA call is involved."""
    assert lib.g4attn_wait_limit_ns() == g4.DEFAULT_WAIT_LIMIT_NS
    try:
        assert lib.g4attn_set_wait_limit_ns(1000) == g4.G4_OK
        assert lib.g4attn_wait_limit_ns() == 1000
        assert lib.g4attn_set_wait_limit_ns(g4.DEFAULT_WAIT_LIMIT_NS + 1) == g4.G4_ERR_INVALID
        assert lib.g4attn_wait_limit_ns() == 1000
        assert lib.g4attn_set_wait_limit_ns(0) == g4.G4_OK
        assert lib.g4attn_wait_limit_ns() == 0
    finally:
        assert lib.g4attn_set_wait_limit_ns(g4.DEFAULT_WAIT_LIMIT_NS) == g4.G4_OK


def test_tensor_parallel_head_slices_are_the_only_other_geometries(lib):
    """A layer descriptor may name one tensor-parallel rank's heads: 32/tp query heads with 16/tp
    (sliding) or max(1, 4/tp) (global) KV heads, tp in {1, 2, 4, 8}; other head counts fail closed.
    The provenance record names the slice's shape. No CUDA call is involved."""
    for tp in (1, 2, 4, 8):
        for layer in (g4.sliding_layer(tp=tp), g4.global_layer(tp=tp)):
            buf = ctypes.create_string_buffer(2048)
            assert lib.g4attn_provenance(ctypes.byref(layer), buf, len(buf)) > 0
            assert f"Hq{layer.n_q_heads},Hkv{layer.n_kv_heads}," in buf.value.decode()
    assert g4.global_layer(tp=8).n_kv_heads == 1 and g4.global_layer(tp=4).n_kv_heads == 1
    for kind, nq, nkv in (("sliding", 16, 16), ("sliding", 8, 2), ("sliding", 2, 1), ("sliding", 64, 32),
                          ("global", 4, 2), ("global", 16, 4), ("global", 2, 1), ("global", 8, 2)):
        layer = g4.sliding_layer() if kind == "sliding" else g4.global_layer()
        layer.n_q_heads, layer.n_kv_heads = nq, nkv
        assert lib.g4attn_provenance(ctypes.byref(layer), None, 0) == -1, (kind, nq, nkv)
        assert lib.g4attn_decode_workspace_bytes(ctypes.byref(layer), 4, 8) == 0
    # the decode workspace scales with the slice's query heads
    full = lib.g4attn_decode_workspace_bytes(ctypes.byref(g4.global_layer()), 4, 100)
    eighth = lib.g4attn_decode_workspace_bytes(ctypes.byref(g4.global_layer(tp=8)), 4, 100)
    assert 0 < eighth < full and abs(8 * eighth - full) <= 8 * 256
