"""The C-ABI library loads and exports every symbol include/rbkv.h declares
(no compute calls: these run without a GPU)."""
import re
import subprocess
from pathlib import Path

import pytest

HEADER = Path(__file__).resolve().parent.parent / "include" / "rbkv.h"


def declared_symbols():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rbkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("rbkv_compose_pass", "rbkv_kv_append", "rbkv_ragged_attention",
                     "rbkv_attention_workspace_bytes", "rbkv_release_seq"):
        assert required in names


def test_library_exports_every_declared_symbol(rbkv):
    L = rbkv.lib()
    for name in declared_symbols():
        assert hasattr(L, name), name
    assert set(declared_symbols()) == set(rbkv.SIGNATURES)
    out = subprocess.run(["nm", "-D", "--defined-only", str(rbkv.library_path())],
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(rbkv_[a-z0-9_]+)\b", out))
    assert set(declared_symbols()) <= exported
    assert L.rbkv_abi_version() == 3


def test_bad_config_is_rejected_without_a_gpu(rbkv):
    import pytest
    with pytest.raises(rbkv.RbkvError):
        rbkv.Composer(rbkv.Config(8, 3, 64, 16, "f32", 10))
    with pytest.raises(rbkv.RbkvError):
        rbkv.Composer(rbkv.Config(8, 2, 48, 16, "f32", 10))
    with pytest.raises(rbkv.RbkvError):
        rbkv.Composer(rbkv.Config(8, 2, 64, 0, "f32", 10))


def test_debug_corrupt_validates_arguments(rbkv):
    c = rbkv.Composer(rbkv.Config(8, 2, 64, 16, "f32", 10))
    p = c.compose(20, 0, [(1, 20, 0)])
    assert len(p.meta.block_ids) == 2 and p.num_tokens == 20
    with pytest.raises(rbkv.RbkvError):
        p.debug_corrupt("block", 2, 0)
    with pytest.raises(rbkv.RbkvError):
        p.debug_corrupt("slot", -1, 0)
    p.debug_corrupt("block", 1, 9)
    p.debug_corrupt("slot", 19, 3)
    assert rbkv.lib().rbkv_debug_corrupt_pass(p._h, 2, 0, 0) == -1   # which: 0 or 1
