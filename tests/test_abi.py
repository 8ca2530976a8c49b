"""The C-ABI library (CPU only, no GPU needed): it builds, loads, exports
every function include/treeverify.h declares, and rejects bad arguments on
the host before touching the GPU."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                 text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    bm = __graft_entry__._build_module()
    if not os.path.exists(bm.LIB) and not shutil.which("nvcc"):
        pytest.skip("library not built and nvcc unavailable")
    return ctypes.CDLL(bm.build())


def test_header_declares_the_four_steps():
    fns = declared_functions()
    for name in ("tree_mask_build", "tree_verify_attention", "tree_accept", "kv_compact",
                 "tree_verify_attention_workspace", "tree_accept_workspace",
                 "tv_status_string", "tv_abi_version"):
        assert name in fns, fns


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    lib.tv_status_string.restype = ctypes.c_char_p
    for code in range(9):
        assert lib.tv_status_string(code)
    assert lib.tv_status_string(99) == b"unknown status"
    assert lib.tv_abi_version() == 2


def test_host_argument_checks_need_no_gpu(lib):
    p = ctypes.c_void_p
    # N outside [1, 64]
    assert lib.tree_mask_build(p(0), 1, 65, None, p(0), p(0), p(0), p(0)) == 1
    assert lib.tree_mask_build(p(0), -1, 4, None, p(0), p(0), p(0), p(0)) == 1
    # B == 0: nothing to do, no launch
    assert lib.tree_mask_build(p(0), 0, 4, None, p(0), p(0), p(0), p(0)) == 0
    # stochastic acceptance needs draft probabilities
    f = lib.tree_accept
    f.argtypes = [ctypes.c_int, p, p, p, p, ctypes.c_int, ctypes.c_int, p, ctypes.c_int,
                  ctypes.c_uint64, ctypes.c_uint64, p, p, p, ctypes.c_int, p, p, ctypes.c_size_t, p]
    nz = p(16)
    assert f(1, nz, nz, nz, None, 2, 4, None, 10, 0, 0, nz, nz, nz, 4, nz, None, 0, None) == 1
    assert f(0, nz, nz, nz, None, 2, 4, None, 0, 0, 0, nz, nz, nz, 4, nz, None, 0, None) == 1
    # attention: head size 96 is not built for bf16 -> unsupported
    a = lib.tree_verify_attention
    a.argtypes = [p, p, p, p, ctypes.c_int, p, p, ctypes.c_int, ctypes.c_int, p] + \
        [ctypes.c_int] * 6 + [ctypes.c_float, p, p, p, ctypes.c_size_t, p]
    assert a(nz, nz, nz, nz, 4, nz, nz, 1, 4, None, 8, 2, 96, 16, 10, 1, 0.0, nz, nz, nz, 1 << 20,
             None) == 4
    # Hq not a multiple of Hkv -> invalid
    assert a(nz, nz, nz, nz, 4, nz, nz, 1, 4, None, 6, 4, 128, 16, 10, 1, 0.0, nz, nz, nz,
             1 << 20, None) == 1
    # kernel count query: rejected shapes -> -1, empty batch -> 0 (no device needed)
    k = lib.tree_verify_attention_kernels
    k.argtypes = [ctypes.c_int] * 8 + [ctypes.c_size_t]
    assert k(1, 4, 6, 4, 128, 10, 16, 1, 0) == -1     # Hq not a multiple of Hkv
    assert k(1, 65, 8, 2, 128, 10, 16, 1, 0) == -1    # more than 64 nodes
    assert k(0, 4, 8, 2, 128, 10, 16, 1, 0) == 0
    # tree_kv_append: host-side argument checks (nothing is launched)
    ap = lib.tree_kv_append
    ap.argtypes = [p, p, p, ctypes.c_int, ctypes.c_int, p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_float, p, p, p, ctypes.c_int, p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, p, p]
    args = lambda B, N, Hkv, d, theta, depth, dt=1: (nz, nz, depth, B, N, None, Hkv, d, theta, nz,
                                                     nz, nz, 4, nz, 16, 10, dt, nz, None)
    assert ap(*args(1, 65, 2, 128, 0.0, nz)) == 1          # more than 64 nodes
    assert ap(*args(1, 4, 2, 127, 0.0, nz)) == 1           # odd head size
    assert ap(*args(1, 4, 2, 4, 0.0, nz)) == 4             # 8-byte rows: not 16-byte vectors
    assert ap(*args(1, 4, 2, 128, 10000.0, None)) == 1     # rotation without depth
    assert ap(*args(1, 4, 2, 128, float("nan"), nz)) == 1  # NaN theta
    assert ap(*args(0, 4, 2, 128, 0.0, nz)) == 0           # empty batch: nothing to do
    assert ap(*args(1, 4, 2, 128, 0.0, nz, dt=7)) == 1     # unknown dtype
    # kv_compact: rows that are not a multiple of 16 bytes -> unsupported
    c = lib.kv_compact
    c.argtypes = [p, p, ctypes.c_int, ctypes.c_int64, p, ctypes.c_int, p, p, p] + \
        [ctypes.c_int] * 7 + [p, p, p, p, p]
    assert c(nz, nz, 1, 0, nz, 4, nz, nz, nz, 4, 2, 2, 12, 16, 10, 1, nz, None, None, nz,
             None) == 4


def test_draft_tree_host_checks(lib):
    p, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    ws = lib.draft_tree_workspace
    ws.restype, ws.argtypes = sz, [ci, ci, ci]
    f = lib.draft_tree_expand
    f.restype = ci
    f.argtypes = [p, p, ci, ci, ci, ci, ci, ci, p, p, p, p, p, p, p, sz, p]
    assert ws(2, 4, 3) > 0 and ws(2, 17, 3) == 0 and ws(0, 4, 3) == 0
    assert ws(1, 16, 8) > 0 and ws(1, 16, 9) == 0           # 1809 / 2065 created nodes
    need = ws(2, 4, 3)
    buf = ctypes.create_string_buffer(need + 32)
    a16 = (ctypes.addressof(buf) + 15) // 16 * 16
    dev = p(0x1000)                                          # never dereferenced on the host

    def call(B=2, V=100, k=4, layer=0, layers=3, N=10, logits=dev, root=dev, parents=dev,
             tokens=dev, status=dev, wsp=p(a16), wsb=need):
        return f(logits, root, B, V, k, layer, layers, N, None, None, parents, tokens, None,
                 status, wsp, wsb, None)

    INVALID, UNSUPPORTED, WORKSPACE = 1, 4, 8
    assert call(k=0) == INVALID and call(k=17) == INVALID and call(k=101) == INVALID
    assert call(V=0) == INVALID and call(V=(1 << 30) + 1) == INVALID
    assert call(layers=0) == INVALID and call(layer=3) == INVALID and call(layer=-1) == INVALID
    assert call(N=0) == INVALID and call(N=65) == INVALID
    assert call(k=1, layers=2, N=4) == INVALID               # only 3 nodes are ever created
    assert call(k=16, layers=10, N=8) == UNSUPPORTED
    assert call(B=-1) == INVALID and call(B=0) == 0
    assert call(logits=None) == INVALID and call(status=None) == INVALID
    assert call(root=None) == INVALID                        # layer 0 reads the root tokens
    assert call(layer=2, parents=None) == INVALID and call(layer=2, tokens=None) == INVALID
    assert call(wsp=None) == WORKSPACE and call(wsp=p(a16 + 4)) == WORKSPACE
    assert call(wsb=need - 1) == WORKSPACE


def test_draft_tree_binding_checks_need_no_gpu(lib):
    """The Python binding rejects wrong dtypes, a row count that does not match
    the layer, and host tensors, before the library is called."""
    torch = pytest.importorskip("torch")
    import eagle_speculative_decoding_parent_gb300 as tv
    st = torch.zeros(2, dtype=torch.int32)
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(TypeError):
        tv.draft_tree_expand(torch.zeros(2, 1, 8, dtype=torch.float64), 0, 2, st, ws, topk=2)
    with pytest.raises(ValueError, match="rows per sequence"):
        tv.draft_tree_expand(torch.zeros(2, 1, 8), 1, 2, st, ws, topk=2)
    with pytest.raises(ValueError, match="CUDA device"):
        tv.draft_tree_expand(torch.zeros(2, 1, 8), 0, 2, st, ws, topk=2,
                             root_tokens=torch.zeros(2, dtype=torch.int32))


def declared_arity():
    """Parameter count of every function include/treeverify.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(([^;{}]*?)\)\s*;", text):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_handles_match_the_header(lib):
    """Each module-level ctypes handle of the binding is the C symbol it is
    named after and carries the header's parameter count: a later rebinding of
    a handle's name (a helper of the same name) fails here, on the CPU."""
    pytest.importorskip("torch")
    import eagle_speculative_decoding_parent_gb300 as tv
    arity = declared_arity()
    handles = {n: getattr(tv, n) for n in dir(tv)
               if isinstance(getattr(tv, n), ctypes._CFuncPtr)}
    bound = {}
    for name, fn in handles.items():
        assert fn.__name__ in arity, (name, fn.__name__)
        assert len(fn.argtypes) == arity[fn.__name__], (name, fn.__name__, len(fn.argtypes))
        bound[fn.__name__] = name
    # every entry point the binding exports has its handle
    for public in ("tree_mask_build", "tree_verify_attention", "tree_verify_attention_noalloc",
                   "tree_accept", "kv_compact", "tree_kv_append", "draft_tree_expand",
                   "draft_tree_workspace", "tree_verify_attention_workspace",
                   "tree_accept_workspace", "tree_verify_attention_kernels"):
        assert public in bound, public
    assert tv._draft_expand.__name__ == "draft_tree_expand" and len(tv._draft_expand.argtypes) == 17


def _attn_host_tensors(torch, dtype=None, mask_dtype=None, status_dtype=None, table_dtype=None,
                       kv_dtype=None):
    B, N, Hq, Hkv, d, nb, bs = 2, 3, 4, 2, 64, 6, 16
    dtype = dtype or torch.bfloat16
    q = torch.zeros(B, N, Hq, d, dtype=dtype)
    k = torch.zeros(nb, Hkv, bs, d, dtype=kv_dtype or dtype)
    v = torch.zeros(nb, Hkv, bs, d, dtype=kv_dtype or dtype)
    bt = torch.zeros(B, 3, dtype=table_dtype or torch.int32)
    P = torch.zeros(B, dtype=torch.int32)
    mask = torch.zeros(B, N, dtype=mask_dtype or torch.int64)
    out = torch.zeros_like(q)
    st = torch.zeros(B, dtype=status_dtype or torch.int32)
    return q, k, v, bt, P, mask, out, st


@pytest.mark.parametrize("entry", ["tree_verify_attention", "tree_verify_attention_noalloc"])
def test_attention_bindings_check_dtypes_and_shapes(lib, entry):
    """Both attention entry points reject, before any pointer reaches the
    library, buffers whose element type or shape would make the kernels index
    past their end (an int32 mask read as 64-bit words, an int8 status written
    as int32, caches of another type than q)."""
    torch = pytest.importorskip("torch")
    import eagle_speculative_decoding_parent_gb300 as tv
    fn = getattr(tv, entry)
    for kw, exc in ((dict(mask_dtype=torch.int32), TypeError),
                    (dict(status_dtype=torch.int8), TypeError),
                    (dict(table_dtype=torch.int64), TypeError),
                    (dict(kv_dtype=torch.float16), TypeError),
                    (dict(kv_dtype=torch.float32), TypeError),
                    (dict(dtype=torch.float16), TypeError)):
        with pytest.raises(exc):
            fn(*_attn_host_tensors(torch, **kw))
    q, k, v, bt, P, mask, out, st = _attn_host_tensors(torch)
    with pytest.raises(ValueError):
        fn(q, k, v, bt, P, mask[:, :2], out, st)          # mask narrower than N
    with pytest.raises(ValueError):
        fn(q, k, v, bt, P, mask, out, st[:1])             # status shorter than B
    with pytest.raises(ValueError):
        fn(q, k, v, bt[:1], P, mask, out, st)             # block table for fewer sequences
    with pytest.raises(ValueError, match="CUDA device"):
        fn(q, k, v, bt, P, mask, out, st)                 # well-formed, but host memory


def test_accept_and_compact_bindings_check_dtypes(lib):
    torch = pytest.importorskip("torch")
    import eagle_speculative_decoding_parent_gb300 as tv
    B, N, V, mp = 2, 4, 10, 3
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32)
    args = lambda **o: dict(dict(mode=tv.GREEDY, parents=i32(B, N), draft_tokens=i32(B, N),
                                 target=torch.zeros(B, N, V), draft_probs=None,
                                 accept_len=i32(B), path=i32(B, mp), out_tokens=i32(B, mp),
                                 status=i32(B)), **o)
    with pytest.raises(TypeError):
        tv.tree_accept(**args(parents=torch.zeros(B, N, dtype=torch.int64)))
    with pytest.raises(ValueError):
        tv.tree_accept(**args(out_tokens=i32(B, mp + 1)))
    with pytest.raises(TypeError):
        tv.tree_accept(**args(status=torch.zeros(B, dtype=torch.int8)))
    with pytest.raises(ValueError, match="CUDA device"):
        tv.tree_accept(**args())
    k = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    cargs = lambda **o: dict(dict(k_cache=k, v_cache=k.clone(), block_table=i32(B, 2),
                                  prefix_lens=i32(B), path=i32(B, mp), accept_len=i32(B),
                                  new_lens=i32(B), status=i32(B)), **o)
    with pytest.raises(TypeError):
        tv.kv_compact(**cargs(v_cache=k.float()))
    with pytest.raises(TypeError):
        tv.kv_compact(**cargs(src_slots=i32(B, mp)))
    with pytest.raises(ValueError):
        tv.kv_compact(**cargs(num_layers=2, layer_stride=k.numel()))
    with pytest.raises(ValueError, match="CUDA device"):
        tv.kv_compact(**cargs())


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_is_plain_c_and_cpp(lang, std, tmp_path):
    """include/treeverify.h compiles on its own as C99 and as C++11, with no
    CUDA header: the boundary carries only plain pointers and sizes."""
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    import subprocess
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-x", lang, HEADER], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
