"""The binding's ctypes structures have exactly the C layout of include/wf.h:
every structure's size and every field's offset are checked by the C
compiler itself (static assertions compiled with gcc, nothing is written to
disk), so a field added on one side only fails here instead of corrupting
calls."""

import ctypes
import os
import shutil
import subprocess

import pytest

import chunk_causal_dit_round_b300 as wf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STRUCTS = [wf.wf_plan_opts, wf.wf_buffer_sizes, wf.wf_round_info, wf.wf_dit_layer, wf.wf_dit_model]


def c_source():
    lines = ['#include "wf.h"', "#include <stddef.h>"]
    for st in STRUCTS:
        name = st.__name__
        lines.append(f'_Static_assert(sizeof({name}) == {ctypes.sizeof(st)}, "sizeof {name}");')
        for fname, _ in st._fields_:
            off = getattr(st, fname).offset
            lines.append(f'_Static_assert(offsetof({name}, {fname}) == {off}, "{name}.{fname}");')
    return "\n".join(lines) + "\n"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_ctypes_structs_match_the_header():
    src = c_source()
    r = subprocess.run(["gcc", "-std=c11", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        "-x", "c", "-"], input=src, capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr[-3000:]


def test_every_field_is_checked():
    """The C structures have no field the binding lacks: the last field's
    offset plus its size reaches the structure's size up to alignment."""
    for st in STRUCTS:
        name, typ = st._fields_[-1]
        end = getattr(st, name).offset + ctypes.sizeof(typ)
        assert ctypes.sizeof(st) - end < ctypes.alignment(st), st.__name__
