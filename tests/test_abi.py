"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol the header declares, and its host-only logic matches the oracle."""
import ctypes
import os
import re

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_layer_gb300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", src)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("dflash_fuse_context", "dflash_inject_kv", "dflash_draft_block",
              "dflash_verify_greedy", "dflash_create", "dflash_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(dfl):
    lib = ctypes.CDLL(dfl.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(dfl.EXPORTED)


@pytest.mark.parametrize("n_t", range(4, 70))
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_layer_ids_match_oracle(dfl, n_t, n):
    try:
        ref = O.build_target_layer_ids(n_t, n)
    except ValueError:
        with pytest.raises(dfl.DFlashError):
            dfl.dflash_build_target_layer_ids(n_t, n)
        return
    assert dfl.dflash_build_target_layer_ids(n_t, n) == ref


def test_strerror_and_argument_errors(dfl):
    assert dfl.dflash_strerror(0) == "ok"
    assert "capacity" in dfl.dflash_strerror(4)
    with pytest.raises(dfl.DFlashError) as e:
        dfl.dflash_build_target_layer_ids(36, 0)
    assert e.value.code == 1
    # null pointers are rejected on the host before any launch
    lib = dfl._lib
    assert lib.dflash_verify_greedy(None, None, 1, 4, None, None, None, None, None, None, None) == 1
    assert lib.dflash_draft_block(None, None, 1, 4, None, None, None, None, None, 0, None) == 1
    assert lib.dflash_fuse_context(None, None, 1, None, None, 0, None) == 1
    assert lib.dflash_draft_round(None, None, 4, None, None, None, None, 1, 4, None, None, None,
                                  None, None, 0, None) == 1
    assert lib.dflash_workspace_bytes(None, 1, 16, 16) == 0


def test_sampling_scratch_and_argument_errors(dfl):
    """The sampling calls' scratch size (per row 16 bytes per 2048-entry
    vocabulary chunk plus 48, and 512) and their host-side argument checks."""
    assert dfl.dflash_sampling_ws_bytes(15, 151936) == 15 * (75 * 16 + 48) + 512
    assert dfl.dflash_sampling_ws_bytes(1, 2048) == 16 + 48 + 512
    assert dfl.dflash_sampling_ws_bytes(1, 2049) == 32 + 48 + 512
    assert dfl.dflash_sampling_ws_bytes(0, 10) == 512
    assert dfl.dflash_sampling_ws_bytes(-1, 10) == 0
    assert dfl.dflash_sampling_ws_bytes(3, 0) == 0
    lib = dfl._lib
    assert lib.dflash_sample_rows(None, None, 1, 16, 1.0, None, None, 0, None, None, 0, None) == 1
    assert lib.dflash_verify_rejection(None, None, None, None, 16, None, None, 1, 4, None, None,
                                       None, None, None, None, None, 0, None) == 1
    assert lib.dflash_lm_head_logits(None, None, 1, None, 0, None, None, 0, None) == 1


def test_round_host_layout_and_argument_errors(dfl):
    """dflash_round_host's result length (ids and tokens [batch, B], then
    accept, tau and bonus [batch] each padded to a multiple of 4) and its
    host-side argument checks, which reject before any copy is queued."""
    assert dfl.dflash_round_out_len(1, 16) == 2 * 16 + 3 * 4
    assert dfl.dflash_round_out_len(4, 8) == 2 * 32 + 3 * 4
    assert dfl.dflash_round_out_len(5, 8) == 2 * 40 + 3 * 8
    assert dfl.dflash_round_out_len(32, 16) == 2 * 512 + 3 * 32
    assert dfl.dflash_round_out_len(0, 16) == -1
    assert dfl.dflash_round_out_len(4, 0) == -1
    lib = dfl._lib
    args = [None] * 19
    args[3], args[11], args[12], args[17] = 16, 1, 16, 0
    assert lib.dflash_round_host(*args) == 1          # no handle, no buffers
    args[3] = -1
    assert lib.dflash_round_host(*args) == 1          # negative pending rows
