"""The C-ABI library builds, loads and exports every entry point declared in
include/dflash.h; host-side argument checks work without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import block_diffusion_speculative_ctx_gb300 as dfl
from block_diffusion_speculative_ctx_gb300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    dbuild.build()
    return dfl.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        with open(h) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(dflash_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_round_entry_points():
    names = declared_functions()
    for n in ("dflash_init", "dflash_prefill", "dflash_draft_block", "dflash_verify", "dflash_generate",
              "dflash_destroy", "dflash_last_error", "dflash_inspect"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", dbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_struct_layouts_match_the_header(tmp_path):
    """sizeof/offsetof of the ABI structs, compiled from the header by gcc,
    equal the ctypes mirrors in the binding."""
    prog = tmp_path / "sz.c"
    prog.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "dflash.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(dflash_config), sizeof(dflash_layer_weights),
         sizeof(dflash_weights), sizeof(dflash_stats), offsetof(dflash_config, rope_theta),
         offsetof(dflash_config, alloc_user), offsetof(dflash_weights, draft_norm),
         offsetof(dflash_config, kv_pool_tokens));
  return 0;
}
""")
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(dfl.dflash_config), ctypes.sizeof(dfl.dflash_layer_weights),
            ctypes.sizeof(dfl.dflash_weights), ctypes.sizeof(dfl.dflash_stats),
            dfl.dflash_config.rope_theta.offset, dfl.dflash_config.alloc_user.offset,
            dfl.dflash_weights.draft_norm.offset, dfl.dflash_config.kv_pool_tokens.offset]
    assert got == want


def _valid_cfg():
    from synth import configs
    return dfl.config_from_workload(configs.get("tiny_f32"), 1, 128)


@pytest.mark.parametrize("field,value,needle", [
    ("head_dim", 96, "head_dim"),
    ("n_kv_heads", 3, "n_kv_heads"),
    ("block_size", 0, "block_size"),
    ("block_size", 33, "block_size"),
    ("mask_token", 1024, "mask_token"),
    ("d_model", 200, "d_model"),
    ("dtype", 7, "dtype"),
    ("max_batch", 0, "max_batch"),
    ("kv_pool_tokens", -64, "kv_pool_tokens"),
    ("kv_pool_tokens", 1 << 40, "kv_pool_tokens"),
])
def test_init_rejects_bad_configs_without_touching_the_gpu(lib, field, value, needle):
    cfg = _valid_cfg()
    setattr(cfg, field, value)
    ws = dfl.dflash_weights()
    tl = (dfl.dflash_layer_weights * 4)()
    dl = (dfl.dflash_layer_weights * 2)()
    ws.target, ws.draft = tl, dl
    ctx = ctypes.c_void_p()
    st = lib.dflash_init(ctypes.byref(cfg), ctypes.byref(ws), None, ctypes.byref(ctx))
    assert st == dfl.DFLASH_E_INVAL and not ctx.value
    assert needle in dfl.dflash_last_error(None)


def test_ctx_layer_id_checks(lib):
    cfg = _valid_cfg()
    cfg.ctx_layer_ids[1] = 4
    ws = dfl.dflash_weights()
    ws.target, ws.draft = (dfl.dflash_layer_weights * 4)(), (dfl.dflash_layer_weights * 2)()
    ctx = ctypes.c_void_p()
    assert lib.dflash_init(ctypes.byref(cfg), ctypes.byref(ws), None, ctypes.byref(ctx)) == dfl.DFLASH_E_INVAL
    assert "ctx_layer_ids" in dfl.dflash_last_error(None)


def test_null_arguments(lib):
    ctx = ctypes.c_void_p()
    assert lib.dflash_init(None, None, None, ctypes.byref(ctx)) == dfl.DFLASH_E_INVAL
    assert lib.dflash_prefill(None, 1, None, None, None) == dfl.DFLASH_E_INVAL
    assert lib.dflash_draft_block(None, None) == dfl.DFLASH_E_INVAL
    assert lib.dflash_verify(None, None, None, None) == dfl.DFLASH_E_INVAL
    assert lib.dflash_draft_block_sampled(None, 1.0, None, None) == dfl.DFLASH_E_INVAL
    assert lib.dflash_verify_sampled(None, 1.0, None, None, None, None) == dfl.DFLASH_E_INVAL
    assert lib.dflash_set_block_size(None, 4) == dfl.DFLASH_E_INVAL
    assert lib.dflash_set_sampling_filter(None, 0, 1.0) == dfl.DFLASH_E_INVAL
    assert lib.dflash_block_size(None) == -1
    lib.dflash_destroy(None)
