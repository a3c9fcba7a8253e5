"""Host-side checks that need no GPU: the library loads, exports every
symbol include/dsa.h declares, and the host-only entry points behave."""
import re
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def test_library_exports_every_declared_symbol(dsa):
    with open(os.path.join(ROOT, "include", "dsa.h")) as f:
        header = f.read()
    declared = set(re.findall(r"DSA_API\s+[\w ]+?\b(dsa_\w+)\(", header))
    assert len(declared) >= 9
    L = dsa.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(dsa.abi.EXPORTS) | (declared - set(dsa.abi.EXPORTS))
    assert set(dsa.abi.EXPORTS) <= declared


def test_share_map_matches_closed_form(dsa):
    full, src, n = dsa.dsa_index_build_share_map([0, 1, 1, 0], 4)
    assert full == [0, -1, -1, 1] and src == [0, 0, 0, 1] and n == 2
    full, src, n = dsa.dsa_index_build_share_map(None, 3, skip_offset=7)
    assert full == [0, 1, 2] and src == [0, 1, 2] and n == 3


@pytest.mark.parametrize("types,code", [([1, 0], -5), ([0, 2], -6)])
def test_share_map_errors(dsa, types, code):
    with pytest.raises(dsa.DSAError) as e:
        dsa.dsa_index_build_share_map(types, len(types))
    assert e.value.rc == code


def test_share_map_agrees_with_oracle(dsa):
    import itertools
    import oracle as O

    names = {0: "full", 1: "shared"}
    for L in range(1, 6):
        for types in itertools.product([0, 1], repeat=L):
            try:
                ofull, osrc, on = O.build_index_share_map([names[t] for t in types], 0, L)
            except O.ShareMapError:
                with pytest.raises(dsa.DSAError):
                    dsa.dsa_index_build_share_map(list(types), L)
                continue
            full, src, n = dsa.dsa_index_build_share_map(list(types), L)
            assert n == on and src == [osrc[i] for i in range(L)]
            assert full == [ofull.get(i, -1) for i in range(L)]


def test_workspace_sizes_are_host_computable(dsa):
    a = dsa.dsa_indexer_workspace_size(32, 32, 8192, 64)
    b = dsa.dsa_indexer_workspace_size(64, 32, 8192, 64)
    assert 0 < a < b
    assert dsa.dsa_indexer_workspace_size(32, 32, 8192, 48) == 0  # unsupported page size


def test_selftest_wait_timeout_validates_on_host(dsa):
    import ctypes

    L = dsa.lib()
    fake = ctypes.c_void_p(16)  # never dereferenced: the arguments are rejected first
    assert L.dsa_selftest_wait_timeout(None, 0, fake) == -1
    assert L.dsa_selftest_wait_timeout(None, 10**11, fake) == -1
    assert L.dsa_selftest_wait_timeout(None, 1000, None) == -1
