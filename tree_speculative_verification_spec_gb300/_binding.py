"""ctypes binding of libspectree.so: one Python function per C-ABI entry point,
with the same name.  Argument marshalling only (torch tensors -> device
pointers, the current CUDA stream -> cudaStream_t); every step of the hot path
runs in the library's kernels.  There is no CPU fallback: when the library
cannot be loaded, every call raises."""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspectree.so")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA, SPEC_ERR_WORKSPACE = 0, 1, 2, 3, 4
SPEC_DEV_BAD_TREE, SPEC_DEV_BAD_TOKEN, SPEC_DEV_CAPACITY, SPEC_DEV_TIMEOUT = 1, 2, 4, 8
SPEC_DEV_BAD_BLOCK, SPEC_DEV_BAD_PATH, SPEC_DEV_BAD_TEMP = 16, 32, 64
SPEC_Q_PER_PARENT, SPEC_Q_PER_CHILD = 0, 1  # layouts of the draft rows
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_ATTN_AUTO, SPEC_ATTN_CUDA_CORE, SPEC_ATTN_TCGEN05 = 0, 1, 2
SPEC_ATTN_NOALLOC_BYTES = 16 << 20  # scratch of spec_tree_attention_noalloc

# C signatures (argument ctypes, return ctype) of every exported entry point
_P, _I, _U32, _U64, _SZ, _F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t,
                               ctypes.c_float)
SIGNATURES = {
    "spec_version": ([], _I),
    "spec_status_string": ([_I], ctypes.c_char_p),
    "spec_dev_status_string": ([_I], ctypes.c_char_p),
    "spec_tree_mask_build": ([_P, _P, _I, _I, _P, _P, _P, _P], _I),
    "spec_attention_workspace_size": ([_I, _I, _I, _I, _I, _I, _I], _SZ),
    "spec_tree_attention": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _SZ,
                             _P, _U32, _P], _I),
    "spec_tree_attention_noalloc": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P,
                                     _P, _U32, _P], _I),
    "spec_verify_workspace_size": ([_I, _I, _I], _SZ),
    "spec_tree_verify_greedy": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P, _P], _I),
    "spec_tree_init": ([_P, _I, _I, _P, _P, _P, _P], _I),
    "spec_tree_expand_level": ([_P, _I, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "spec_tree_merge": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P], _I),
    "spec_dsd_optimal_k": ([_P, _P, _I, _I, _P, _P], _I),
    "spec_dsd_select_k": ([_P, _P, _I, _I, _P], _I),
    "spec_dsd_update": ([_P, _P, _I, _I, _I, _I, ctypes.c_double, ctypes.c_double, ctypes.c_double], _I),
    "spec_dsd_graph_keys": ([_I, _I, _P, _P, _I, _P], _I),
    "spec_tree_verify_stochastic": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P, _P], _I),
    "spec_kv_append": ([_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "spec_kv_commit": ([_P, _P, _P, _I, _I, _I, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "spec_kv_commit_layers": ([_P, _P, _I, _P, _I, _I, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P],
                              _I),
    "spec_philox_uniforms": ([_U64, _U32, _P, _I, _I, _P, _P], _I),
    "spec_selftest_bounded_wait": ([_P, _U32, _P], _I),
    "spec_selftest_exp": ([_U32, ctypes.c_longlong, _P, _P, _P], _I),
    "spec_selftest_fx": ([_P, ctypes.c_longlong, _I, _P, _P, _P, _P], _I),
    "spec_selftest_resid": ([_P, _P, _P, ctypes.c_longlong, _P, _P, _P, _P], _I),
}

_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} returned {code} ({status_string(code)})")


def lib():
    """Load libspectree.so (raises when it is missing: no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "tree_speculative_verification_spec_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_string(code):
    return lib().spec_status_string(int(code)).decode()


def spec_dev_status_string(bit):
    return lib().spec_dev_status_string(int(bit)).decode()


def dev_status_names(word):
    """The names of the SPEC_DEV_* bits set in a status word."""
    return [spec_dev_status_string(1 << i) for i in range(31) if int(word) >> i & 1]


def version():
    return lib().spec_version()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, code):
    if code != SPEC_OK:
        raise SpecError(fn, code)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def spec_tree_mask_build(parent, tree_off, B, n_max, mask, depth, status, stream=None):
    _check("spec_tree_mask_build", lib().spec_tree_mask_build(
        _ptr(parent), _ptr(tree_off), B, n_max, _ptr(mask), _ptr(depth), _ptr(status), _stream(stream)))


def spec_attention_workspace_size(B, T, n_max, max_prefix, Hq, Hkv, D):
    return int(lib().spec_attention_workspace_size(B, T, n_max, max_prefix, Hq, Hkv, D))


def spec_tree_attention(q, k_cache, v_cache, block_table, max_blocks, block_size, num_blocks, prefix_len, tree_off,
                        mask, B, T, n_max, max_prefix, Hq, Hkv, D, scale, out, workspace, status,
                        flags=SPEC_ATTN_AUTO, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("spec_tree_attention", lib().spec_tree_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_blocks, block_size, num_blocks,
        _ptr(prefix_len), _ptr(tree_off), _ptr(mask), B, T, n_max, max_prefix, Hq, Hkv, D, _dtype_code(q),
        float(scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(status), flags, _stream(stream)))


def spec_tree_attention_noalloc(q, k_cache, v_cache, block_table, max_blocks, block_size, num_blocks, prefix_len,
                                tree_off, mask, B, T, n_max, max_prefix, Hq, Hkv, D, scale, out, status,
                                flags=SPEC_ATTN_AUTO, stream=None):
    _check("spec_tree_attention_noalloc", lib().spec_tree_attention_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_blocks, block_size, num_blocks,
        _ptr(prefix_len), _ptr(tree_off), _ptr(mask), B, T, n_max, max_prefix, Hq, Hkv, D, _dtype_code(q),
        float(scale), _ptr(out), _ptr(status), flags, _stream(stream)))


def spec_verify_workspace_size(B, n_max, V):
    return int(lib().spec_verify_workspace_size(B, n_max, V))


def spec_tree_verify_greedy(p_logits, tokens, parent, tree_off, B, n_max, V, path, accept_len, emitted, n_emitted,
                            workspace, status, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("spec_tree_verify_greedy", lib().spec_tree_verify_greedy(
        _ptr(p_logits), _ptr(tokens), _ptr(parent), _ptr(tree_off), B, n_max, V,
        _ptr(path), _ptr(accept_len), _ptr(emitted), _ptr(n_emitted), _ptr(workspace), ws_bytes, _ptr(status),
        _stream(stream)))


def spec_tree_verify_stochastic(p_logits, q_probs, tokens, parent, tree_off, uniforms, B, n_max, V, path,
                                accept_len, emitted, n_emitted, workspace, status, stream=None, inv_temp=None,
                                q_layout=SPEC_Q_PER_PARENT):
    """inv_temp: float32 device tensor [B] of inverse temperatures, or None
    (1); q_layout: SPEC_Q_PER_PARENT or SPEC_Q_PER_CHILD."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("spec_tree_verify_stochastic", lib().spec_tree_verify_stochastic(
        _ptr(p_logits), _ptr(q_probs), _ptr(tokens), _ptr(parent), _ptr(tree_off), _ptr(uniforms), _ptr(inv_temp),
        q_layout, B, n_max, V,
        _ptr(path), _ptr(accept_len), _ptr(emitted), _ptr(n_emitted), _ptr(workspace), ws_bytes, _ptr(status),
        _stream(stream)))


def spec_tree_init(root_tok, B, n_total, tree_off, parent, tokens, stream=None):
    _check("spec_tree_init", lib().spec_tree_init(_ptr(root_tok), B, n_total, _ptr(tree_off), _ptr(parent),
                                                  _ptr(tokens), _stream(stream)))


def spec_tree_expand_level(scores, B, F, V, k, level_start, n_total, parent, tokens, stream=None):
    _check("spec_tree_expand_level", lib().spec_tree_expand_level(
        _ptr(scores), B, F, V, k, level_start, n_total, _ptr(parent), _ptr(tokens), _stream(stream)))


def spec_tree_merge(seqs, lens, root_tok, B, M, m, V, tree_off, parent, tokens, src, node_of, status, stream=None):
    _check("spec_tree_merge", lib().spec_tree_merge(
        _ptr(seqs), _ptr(lens), _ptr(root_tok), B, M, m, V, _ptr(tree_off), _ptr(parent), _ptr(tokens), _ptr(src),
        _ptr(node_of), _ptr(status), _stream(stream)))


def _hptr(a, dtype):
    """Host (numpy) array argument: C-contiguous and of the C type, else an error."""
    import numpy as np
    if a is None:
        return None
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise ValueError(f"host arguments must be C-contiguous numpy arrays of {np.dtype(dtype).name}")
    return a.ctypes.data_as(ctypes.c_void_p)


def spec_dsd_optimal_k(al, itl, k_values, k_opt):
    """al, itl: float64 [n_bs, n_k]; k_values int32 [n_k]; k_opt int32 [n_bs] out (host arrays)."""
    import numpy as np
    n_bs, n_k = al.shape
    _check("spec_dsd_optimal_k", lib().spec_dsd_optimal_k(_hptr(al, np.float64), _hptr(itl, np.float64), n_bs, n_k,
                                                          _hptr(k_values, np.int32), _hptr(k_opt, np.int32)))


def spec_dsd_select_k(bs_table, k_table, bs):
    import numpy as np
    out = np.zeros(1, np.int32)
    _check("spec_dsd_select_k", lib().spec_dsd_select_k(_hptr(bs_table, np.int32), _hptr(k_table, np.int32),
                                                        len(bs_table), int(bs), _hptr(out, np.int32)))
    return int(out[0])


def spec_dsd_update(al, itl, bs_index, k_index, al_sample, itl_sample, weight):
    import numpy as np
    n_bs, n_k = al.shape
    _check("spec_dsd_update", lib().spec_dsd_update(_hptr(al, np.float64), _hptr(itl, np.float64), n_bs, n_k,
                                                    bs_index, k_index, al_sample, itl_sample, weight))


def spec_dsd_graph_keys(max_tokens, max_k):
    """Returns [(tokens, K), ...]."""
    import numpy as np
    cnt = np.zeros(1, np.int32)
    _check("spec_dsd_graph_keys", lib().spec_dsd_graph_keys(max_tokens, max_k, None, None, 0, _hptr(cnt, np.int32)))
    n = int(cnt[0])
    t, k = np.zeros(max(n, 1), np.int32), np.zeros(max(n, 1), np.int32)
    _check("spec_dsd_graph_keys", lib().spec_dsd_graph_keys(max_tokens, max_k, _hptr(t, np.int32),
                                                            _hptr(k, np.int32), n, _hptr(cnt, np.int32)))
    return list(zip(t[:n].tolist(), k[:n].tolist()))


def spec_kv_append(k_new, v_new, k_cache, v_cache, block_table, max_blocks, block_size, num_blocks, prefix_len,
                   tree_off, B, n_max, Hkv, D, status, stream=None):
    """k_new / v_new: [T][Hkv][D] CUDA tensors of the caches' dtype."""
    if k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype:
        raise ValueError("k_new / v_new must have the caches' dtype")
    _check("spec_kv_append", lib().spec_kv_append(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_blocks, block_size,
        num_blocks, _ptr(prefix_len), _ptr(tree_off), B, n_max, Hkv, D, _dtype_code(k_cache), _ptr(status),
        _stream(stream)))


def spec_kv_commit(k_cache, v_cache, block_table, max_blocks, block_size, num_blocks, prefix_len, path, path_stride,
                   accept_len, B, Hkv, D, new_len, status, stream=None):
    _check("spec_kv_commit", lib().spec_kv_commit(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_blocks, block_size, num_blocks, _ptr(prefix_len),
        _ptr(path), path_stride, _ptr(accept_len), B, Hkv, D, _dtype_code(k_cache), _ptr(new_len), _ptr(status),
        _stream(stream)))


def spec_kv_commit_layers(k_ptrs, v_ptrs, layers, block_table, max_blocks, block_size, num_blocks, prefix_len, tree_off,
                          path, path_stride, accept_len, B, Hkv, D, dtype, new_len, free_pool, free_count, status,
                          stream=None):
    """k_ptrs / v_ptrs: int64 device tensors of the layers' cache addresses;
    dtype: SPEC_F32 or SPEC_BF16; free_pool / free_count: int32 device
    tensors, or None for a commit without release."""
    cap = 0 if free_pool is None else free_pool.numel()
    _check("spec_kv_commit_layers", lib().spec_kv_commit_layers(
        _ptr(k_ptrs), _ptr(v_ptrs), layers, _ptr(block_table), max_blocks, block_size, num_blocks, _ptr(prefix_len),
        _ptr(tree_off), _ptr(path), path_stride, _ptr(accept_len), B, Hkv, D, dtype, _ptr(new_len), _ptr(free_pool),
        cap, _ptr(free_count), _ptr(status), _stream(stream)))


def spec_philox_uniforms(seed, round_, tree_off, B, n_max, out, stream=None):
    _check("spec_philox_uniforms", lib().spec_philox_uniforms(
        ctypes.c_uint64(seed), ctypes.c_uint32(round_), _ptr(tree_off), B, n_max, _ptr(out), _stream(stream)))


def spec_selftest_bounded_wait(status, polls, stream=None):
    _check("spec_selftest_bounded_wait", lib().spec_selftest_bounded_wait(_ptr(status), ctypes.c_uint32(polls),
                                                                            _stream(stream)))


def spec_selftest_exp(first_bits, n, exp_scalar=None, exp_pair=None, stream=None):
    """exp_scalar / exp_pair: float32 CUDA tensors of n entries (or None)."""
    _check("spec_selftest_exp", lib().spec_selftest_exp(ctypes.c_uint32(first_bits), n, _ptr(exp_scalar),
                                                        _ptr(exp_pair), _stream(stream)))


def spec_selftest_fx(v, seg, fx_out=None, seg_scalar=None, seg_pair=None, stream=None):
    """v: float32 CUDA tensor; outputs: int64 CUDA tensors (raw uint64 bits) or None."""
    _check("spec_selftest_fx", lib().spec_selftest_fx(_ptr(v), v.numel(), seg, _ptr(fx_out), _ptr(seg_scalar),
                                                      _ptr(seg_pair), _stream(stream)))


def spec_selftest_resid(d, q, Zp, r_div=None, r_markstein=None, r_pair=None, stream=None):
    """d, q: float32 CUDA tensors of n entries; Zp: ceil(n / 2) normalisers."""
    _check("spec_selftest_resid", lib().spec_selftest_resid(_ptr(d), _ptr(q), _ptr(Zp), d.numel(), _ptr(r_div),
                                                            _ptr(r_markstein), _ptr(r_pair), _stream(stream)))
