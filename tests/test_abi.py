"""C-ABI boundary checks that need no GPU: the library builds and loads,
exports every function include/kvs.h declares, the binding's structures
match the C layouts, and configuration checks / size arithmetic work."""
import ctypes
import re
import subprocess
from pathlib import Path

import pytest

import paged_kv_cache_flash_gb300 as K
from paged_kv_cache_flash_gb300 import build as B

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "kvs.h"


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def _declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(kvs_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(names) == set(K.exported_symbols())


def test_struct_layouts_match_header(tmp_path):
    src = tmp_path / "sz.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "kvs.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\","
        "sizeof(kvs_config), sizeof(kvs_sizes), sizeof(kvs_buffers), sizeof(kvs_key),"
        "sizeof(kvs_record), sizeof(kvs_gather_args), sizeof(kvs_gather_result),"
        "offsetof(kvs_record, prio), offsetof(kvs_record, mass), offsetof(kvs_record, lrfu));return 0;}\n")
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", str(ROOT / "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    exp = [ctypes.sizeof(K.kvs_config), ctypes.sizeof(K.kvs_sizes), ctypes.sizeof(K.kvs_buffers),
           ctypes.sizeof(K.kvs_key), K.RECORD_DTYPE.itemsize, ctypes.sizeof(K.kvs_gather_args),
           ctypes.sizeof(K.kvs_gather_result), K.RECORD_DTYPE.fields["prio"][1],
           K.RECORD_DTYPE.fields["mass"][1], K.RECORD_DTYPE.fields["lrfu"][1]]
    assert got == exp


def test_record_layout_agrees_with_oracle_restatement():
    import oracle as O
    for name, ofield in [("seq_id", "seq_id"), ("block_idx", "block_idx"), ("score", "score"),
                         ("last_touch", "last_touch"), ("count", "count"), ("tier", "tier"),
                         ("flags", "flags"), ("prio", "prio"), ("mass", "mass"), ("lrfu", "lrfu")]:
        assert K.RECORD_DTYPE.fields[name][1] == O.REC_DTYPE.fields[ofield][1]
        assert K.RECORD_DTYPE.fields[name][0] == O.REC_DTYPE.fields[ofield][0]


def test_fp8_pages_are_half_size(lib):
    cfg = K.make_config(80, 64, 8, 128, pool_blocks=16, max_seqs=1, max_blocks_per_seq=16,
                        kv_dtype=K.KVS_KV_FP8_E4M3)
    assert K.kvs_required_sizes(cfg).page_bytes == 5 * 2**20 // 2


def test_required_sizes_llama70b(lib):
    cfg = K.make_config(80, 64, 8, 128, pool_blocks=8200, max_seqs=1, max_blocks_per_seq=8197)
    sz = K.kvs_required_sizes(cfg)
    assert sz.page_bytes == 5 * 2**20
    assert sz.pool_bytes == 8200 * 5 * 2**20
    assert sz.records_bytes == 8197 * 64
    assert sz.table_bytes == 8197 * 4
    assert sz.staging_bytes == 16 * 5 * 2**20
    assert sz.workspace_bytes > 0


@pytest.mark.parametrize("bad", [
    dict(d=96), dict(Hq=12, Hkv=8), dict(Hq=32, Hkv=2), dict(pool_blocks=0),
    dict(alpha=1.5), dict(cuts=(0.7, 0.6)),
])
def test_config_validation(lib, bad):
    args = dict(L=2, Hq=8, Hkv=2, d=64, pool_blocks=17, max_seqs=1, max_blocks_per_seq=18)
    kw = {}
    for k in ("alpha", "cuts"):
        if k in bad:
            kw[k] = bad.pop(k)
    args.update(bad)
    cfg = K.make_config(**args, **kw)
    with pytest.raises(K.KvsError) as e:
        K.kvs_required_sizes(cfg)
    assert e.value.code == K.KVS_EINVAL


def test_block_tokens_must_be_16(lib):
    cfg = K.make_config(2, 8, 2, 64, 17, 1, 18)
    cfg.block_tokens = 8
    with pytest.raises(K.KvsError):
        K.kvs_required_sizes(cfg)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(K, "LIB_PATH", tmp_path / "missing.so")
    monkeypatch.setattr(K, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        K.lib()
