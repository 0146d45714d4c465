"""The C ABI header is plain C, and the ctypes mirrors in the binding have the header's
struct layouts (field offsets and sizes), checked by compiling a C probe with gcc."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

ATTN_FIELDS = ["q", "cu_seqlens_q", "seq_len", "k_pool", "v_pool", "n_pool_pages", "page_table", "page_logical",
               "n_pages", "head_class", "window", "sink", "B", "Hq", "Hkv", "d", "P", "max_pages", "total_q", "max_q",
               "scale", "out", "lse", "status", "flags", "k_new", "v_new", "k_rot", "rot_coef", "n_rot", "rot_style"]
APPEND_FIELDS = ["k_new", "v_new", "pos", "k_pool", "v_pool", "n_pool_pages", "page_table", "page_logical", "n_pages",
                 "B", "Hkv", "d", "P", "max_pages", "status"]
RING_FIELDS = ["pos", "page_table", "page_logical", "n_pages", "ring", "window", "sink", "B", "Hkv", "P", "max_pages",
               "status", "src_page_table", "src_page_logical"]
ROPE_FIELDS = ["k_src", "n_src_pages", "k_dst", "n_dst_pages", "src_tables", "n_src_entries", "dst_tables",
               "n_dst_entries", "runs", "n_runs", "max_tok", "P", "d", "theta", "style", "status"]
RUN_FIELDS = ["src_tab_off", "src_tab_len", "dst_tab_off", "dst_tab_len", "pos_off0", "pos_on0", "n_tok", "reserved"]


def _probe(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "rk_api.h"', "int main(void) {"]
    for struct, fields in (("rk_attn_args", ATTN_FIELDS), ("rk_rope_args", ROPE_FIELDS), ("rk_rope_run", RUN_FIELDS),
                           ("rk_append_args", APPEND_FIELDS), ("rk_ring_args", RING_FIELDS)):
        lines.append('  printf("%s sizeof %%zu\\n", sizeof(%s));' % (struct, struct))
        for f in fields:
            lines.append('  printf("%s %s %%zu\\n", offsetof(%s, %s));' % (struct, f, struct, f))
    lines += ["  return 0;", "}"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "probe"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr        # the header compiles as C99
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    return {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l}


def test_ctypes_mirrors_match_the_c_header(tmp_path):
    from head_aware_paged_rope_b300 import build as b
    b.build()                                   # the binding loads librk.so when imported
    import head_aware_paged_rope_b300._binding as B
    got = _probe(tmp_path)
    for struct, cls, fields in (("rk_attn_args", B.AttnArgs, ATTN_FIELDS), ("rk_rope_args", B.RopeArgs, ROPE_FIELDS),
                                ("rk_rope_run", B.RopeRun, RUN_FIELDS), ("rk_append_args", B.AppendArgs, APPEND_FIELDS),
                                ("rk_ring_args", B.RingArgs, RING_FIELDS)):
        assert [n for n, _ in cls._fields_] == fields, struct
        assert ctypes.sizeof(cls) == got[(struct, "sizeof")], struct
        for f in fields:
            assert getattr(cls, f).offset == got[(struct, f)], (struct, f)
