"""The C-ABI library loads and exports every symbol include/tg.h declares (no GPU calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tg_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_named_calls():
    names = declared_functions()
    for n in ("tg_build_pages", "tg_compact_topk", "tg_split_map", "tg_decode_attn", "tg_page_score_topk"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib._build.LIB)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_binding_names_match_header(lib):
    for n in declared_functions():
        if n in ("tg_last_error_string",):
            continue
        assert hasattr(lib, n), n


def test_version_and_error_string(lib):
    assert lib.tg_version() >= 100
    with pytest.raises(lib.TGError) as e:
        lib.tg_split_map([[1, 2, 3]], 1)
    assert "N_CTA" in str(e.value)


def test_struct_sizes_match_header(lib):
    assert lib.WORK_ITEM_DTYPE.itemsize == 48
    assert lib._HEADER_DTYPE.itemsize == 80


def test_compact_chunk_workspace_size_and_short_workspace_refused(lib):
    """tg_compact_chunk_workspace: 8 bytes of (slot, chunk position) per head and chunk token,
    then a count per head (256-byte aligned sections).  A workspace one byte short is refused
    on the host, before anything is launched (the pointers below are never dereferenced)."""
    batch, H, C = 3, 8, 100
    need = lib.tg_compact_chunk_workspace(batch, H, C)
    rows = batch * H
    assert need == -(-(-(-rows * C * 8 // 256) * 256 + rows * 4) // 256) * 256
    so = lib.load()
    fake = ctypes.c_void_p(4096)  # 16-byte aligned, never read: the size check comes first
    rc = so.tg_compact_chunk(None, batch, H, 2, 16, 128, 0, C, fake, fake, fake, fake, fake, fake, fake, fake,
                             1, fake, fake, fake, 64, fake, need - 1, None)
    assert rc == -4  # TG_ERR_CAPACITY
    assert b"workspace" in so.tg_last_error_string()
    with pytest.raises(lib.TGError):
        lib.tg_compact_chunk_workspace(batch, 0, C)


def test_compact_topk_workspace_size_and_short_workspace_refused(lib):
    """tg_compact_topk_workspace: per row T, need_eq, two unused ints, then (keys > T, keys == T)
    for every block of 1024 positions.  A workspace one byte short is refused on the host
    (TG_ERR_CAPACITY), before any launch; the pointers below are never dereferenced."""
    batch, H, Nmax = 3, 8, 5000
    need = lib.tg_compact_topk_workspace(batch, H, Nmax)
    assert need == batch * H * (4 + 2 * -(-Nmax // 1024)) * 4
    so = lib.load()
    fake = ctypes.c_void_p(4096)
    rc = so.tg_compact_topk(None, batch, H, 2, 16, 128, Nmax, fake, fake, fake, fake, fake, fake, fake, fake, 1,
                            fake, None, fake, need - 1, None)
    assert rc == -4  # TG_ERR_CAPACITY
    assert b"workspace" in so.tg_last_error_string()
    rc = so.tg_compact_topk(None, batch, H, 2, 16, 128, Nmax, fake, fake, fake, fake, fake, fake, fake, fake, 1,
                            fake, None, None, need, None)
    assert rc == -1  # TG_ERR_INVALID_ARG: no workspace
    with pytest.raises(lib.TGError):
        lib.tg_compact_topk_workspace(batch, H, 0)
    # sizes whose products leave int32 are refused as shapes (TG_ERR_SHAPE), also before any launch
    big = lib.tg_compact_topk_workspace(1, 1, 2**31 - 1)
    assert big == (4 + 2 * 2**21) * 4
    rc = so.tg_compact_topk(None, 2**16, 2**15, 2, 16, 128, Nmax, fake, fake, fake, fake, fake, fake, fake, fake,
                            1, fake, None, fake, 2**62, None)
    assert rc == -2 and b"batch * H" in so.tg_last_error_string()
    rc = so.tg_compact_topk(None, 1, 2, 2, 16, 128, 2**31 - 1, fake, fake, fake, fake, fake, fake, fake, fake,
                            1, fake, None, fake, 2**62, None)
    assert rc == -2 and b"Nmax" in so.tg_last_error_string()


def test_tier_promote_background_checks_arguments_on_the_host(lib):
    """tg_tier_promote_background takes tg_tier_promote's arguments and refuses the same bad
    ones before any launch: sizes out of range and NULL pointers."""
    so = lib.load()
    fake = ctypes.c_void_p(4096)
    # K > n_pages
    rc = so.tg_tier_promote_background(None, 1, fake, 0, fake, 1, 2, 4, 8, fake, fake, fake, fake, fake, 32, fake, 8,
                                       fake, None, None)
    assert rc == -1 and b"tg_tier_promote_background" in so.tg_last_error_string()
    # a NULL selection
    rc = so.tg_tier_promote_background(None, 1, fake, 0, fake, 1, 2, 8, 4, None, fake, fake, fake, fake, 32, fake, 8,
                                       fake, None, None)
    assert rc == -1 and b"NULL" in so.tg_last_error_string()
