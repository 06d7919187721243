"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/spectree.h declares, the binding covers each of them under the same
name, host-side argument checks return their codes before any launch, and the
product shares no code with the oracle."""
import ctypes
import os
import re
import subprocess

import pytest

import tree_speculative_verification_spec_gb300 as S
from tree_speculative_verification_spec_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libpath():
    return build.build()


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("spec_tree_mask_build", "spec_tree_attention", "spec_tree_verify_greedy", "spec_tree_verify_stochastic",
              "spec_kv_commit", "spec_philox_uniforms"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.check_output(["nm", "-D", "--defined-only", libpath]).decode()
    exported = set(re.findall(r"\sT\s+(\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(libpath):
    for n in _declared():
        assert n in _binding.SIGNATURES, n
        if n not in ("spec_version", "spec_status_string"):
            assert callable(getattr(_binding, n)), n
    L = S.lib()
    for n in _declared():
        assert getattr(L, n) is not None


def test_version_and_status_strings(libpath):
    assert S.version() >= 1
    assert S.status_string(0) == "ok"
    assert S.spec_dev_status_string(S.SPEC_DEV_BAD_TEMP) == "bad inverse temperature"
    assert S.spec_dev_status_string(3) == "unknown status bit"
    assert S.dev_status_names(S.SPEC_DEV_BAD_TREE | S.SPEC_DEV_BAD_PATH) == ["bad tree", "bad commit path"]
    assert "workspace" in S.status_string(4)


def test_host_argument_checks_return_codes_without_launching(libpath):
    L = S.lib()
    # negative batch, n_max above the cap
    assert L.spec_tree_mask_build(None, None, -1, 4, None, None, None, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_mask_build(None, None, 1, 2048, None, None, None, None) == S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_mask_build(None, None, 0, 4, None, None, None, None) == S.SPEC_OK  # empty batch: no launch
    assert L.spec_tree_mask_build(None, None, 2, 4, None, None, None, None) == S.SPEC_ERR_INVALID_ARG  # NULL pointers
    # attention: head dim, GQA divisibility, page size, dtype, flags
    args = [None] * 4 + [1, 16, 1] + [None] * 3
    assert L.spec_tree_attention(*args, 1, 1, 4, 10, 4, 2, 96, 1, 0.1, None, None, 0, None, 0, None) == \
        S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_attention(*args, 1, 1, 4, 10, 6, 4, 64, 1, 0.1, None, None, 0, None, 0, None) == \
        S.SPEC_ERR_INVALID_ARG
    args_bs = [None] * 4 + [1, 24, 1] + [None] * 3
    assert L.spec_tree_attention(*args_bs, 1, 1, 4, 10, 4, 2, 64, 1, 0.1, None, None, 0, None, 0, None) == \
        S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_attention(*args, 1, 1, 4, 10, 4, 2, 64, 7, 0.1, None, None, 0, None, 0, None) == \
        S.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_attention(*args, 1, 1, 4, 10, 4, 2, 64, 0, 0.1, None, None, 0, None, 2, None) == \
        S.SPEC_ERR_UNSUPPORTED  # tcgen05 forced on fp32
    assert L.spec_tree_attention(*args, 1, 1, 4, 10, 4, 2, 64, 1, 0.1, None, None, 0, None, 9, None) == \
        S.SPEC_ERR_INVALID_ARG
    # verify: vocabulary above 2^17, NULL pointers
    v = [None] * 6
    assert L.spec_tree_verify_greedy(*v[:4], 1, 4, 200000, None, None, None, None, None, 0, None, None) == \
        S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_verify_greedy(*v[:4], 1, 4, 1000, None, None, None, None, None, 0, None, None) == \
        S.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_verify_stochastic(*v, None, 0, 1, 4, 0, None, None, None, None, None, 0, None, None) == \
        S.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_verify_stochastic(*v, None, 2, 1, 4, 1000, None, None, None, None, None, 0, None, None) == \
        S.SPEC_ERR_INVALID_ARG  # unknown draft-row layout
    # commit: head dim, page size
    assert L.spec_kv_commit(None, None, None, 4, 16, 4, None, None, 4, None, 1, 2, 80, 1, None, None, None) == \
        S.SPEC_ERR_UNSUPPORTED
    assert L.spec_kv_commit(None, None, None, 4, 12, 4, None, None, 4, None, 1, 2, 64, 1, None, None, None) == \
        S.SPEC_ERR_UNSUPPORTED
    assert L.spec_philox_uniforms(0, 0, None, -1, 4, None, None) == S.SPEC_ERR_INVALID_ARG
    # layered commit: layers, page size, pool arguments given by halves
    lc = [None, None, 0, None, 4, 16, 4, None, None, None, 4, None, 1, 2, 64, 1, None, None, 0, None, None, None]
    assert L.spec_kv_commit_layers(*lc) == S.SPEC_ERR_INVALID_ARG  # no layers
    lc[2] = 2
    lc[5] = 12
    assert L.spec_kv_commit_layers(*lc) == S.SPEC_ERR_UNSUPPORTED  # page size not a power of two
    # tree construction: k above 32, a level past n_total, merge shapes past 1023 candidates
    assert L.spec_tree_expand_level(None, 1, 1, 100, 33, 0, 64, None, None, None) == S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_expand_level(None, 1, 2, 100, 4, 0, 9, None, None, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_expand_level(None, 1, 1, 100, 4, 0, 5, None, None, None) == S.SPEC_ERR_INVALID_ARG  # NULLs
    assert L.spec_tree_init(None, 2, 0, None, None, None, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_init(None, 2, 2000, None, None, None, None) == S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_merge(None, None, None, 1, 32, 32, 10, None, None, None, None, None, None, None) == \
        S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_merge(None, None, None, 1, 4, 4, 10, None, None, None, None, None, None, None) == \
        S.SPEC_ERR_INVALID_ARG
    assert L.spec_selftest_bounded_wait(None, 16, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_selftest_bounded_wait(ctypes.c_void_p(16), 0, None) == S.SPEC_ERR_INVALID_ARG


def test_workspace_sizes(libpath):
    a = S.spec_attention_workspace_size(8, 512, 64, 2048, 32, 8, 128)
    assert a >= 256 and a == S.spec_attention_workspace_size(8, 512, 64, 2048, 32, 8, 128)
    # one request with a long prefix needs key splits: room for the partial rows
    one = S.spec_attention_workspace_size(1, 40, 40, 100000, 32, 8, 128)
    assert one >= 2 * 40 * 32 * (128 + 2) * 4
    # room for every node's row statistics (16 bytes per node), at least 256 bytes
    assert S.spec_verify_workspace_size(8, 64, 32000) == 8 * 64 * 16
    assert S.spec_verify_workspace_size(1, 4, 32000) == 256
    assert S.spec_verify_workspace_size(1, 1024, 131072) == 1024 * 16


def test_product_and_oracle_share_no_code(libpath):
    """The product never imports, links or loads the oracle, and the oracle
    never includes the library's headers."""
    pkg = os.path.join(ROOT, "tree_speculative_verification_spec_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "liboracle" not in text and "oracle.c" not in text, f
    needed = subprocess.check_output(["readelf", "-d", libpath]).decode()
    assert "oracle" not in needed
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert "spectree" not in src and "#include \"" not in src
