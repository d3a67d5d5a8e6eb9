"""The boundary as a C program sees it, without a GPU: include/headcast.h
compiles as strict C99, a C program links against libheadcast.so, its host
calls answer like the Python binding's, and every struct the binding mirrors
has the same size and field offsets on both sides."""
import ctypes as C
import os
import subprocess

import pytest

import head_routed_kv_classify_b300 as hc
from head_routed_kv_classify_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.dirname(hc.LIB_PATH)
LABELS_720P = [0, 0, 1, 1, 1, 2, 2, 2, 2, 3, 3, 3]

# Each C struct the binding mirrors, with the binding's field names.
STRUCTS = {
    "hc_config": [name for name, _ in hc.HcConfig._fields_],
    "hc_cache_info": [name for name, _ in hc.HcCacheInfo._fields_],
    "hc_work_item": list(hc.WORK_ITEM_DTYPE.names),
}

PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "headcast.h"

static void layout(void) {
%(layout)s
}

int main(void) {
  hc_config cfg;
  hc_cache_info info;
  hc_work_item items[2048];
  int8_t labels[12] = {%(labels)s};
  size_t bytes = 0;
  int32_t n = 0;
  hc_status st;
  layout();
  printf("abi %%d\n", (int)hc_abi_version());
  if (hc_config_default(&cfg) != HC_OK) return 1;
  cfg.n_heads = 12;
  cfg.head_dim = 128;
  cfg.frame_h = 45;
  cfg.frame_w = 80;
  cfg.frames_per_block = 3;
  cfg.window_frames = 21;
  cfg.dtype = HC_BF16;
  printf("validate %%d\n", (int)hc_config_validate(&cfg));
  st = hc_cache_bytes(&cfg, labels, &bytes);
  printf("cache_bytes %%d %%zu\n", (int)st, bytes);
  st = hc_cache_plan_info(&cfg, labels, &info);
  printf("plan_info %%d %%d %%lld\n", (int)st, (int)info.n_work_items, (long long)info.planned_span);
  st = hc_cache_plan_items(&cfg, labels, NULL, 0, &n);
  printf("plan_count %%d %%d\n", (int)st, (int)n);
  st = hc_cache_plan_items(&cfg, labels, items, 2048, &n);
  printf("plan_items %%d\n", (int)st);
  printf("item0 %%d %%d %%d %%d %%lld %%lld %%d\n", (int)items[0].head, (int)items[0].kind, (int)items[0].q0,
         (int)items[0].nq, (long long)items[0].k_row0, (long long)items[0].k_len, (int)items[0].cta);
  printf("item_last_cta %%d\n", (int)items[n - 1].cta);
  cfg.head_dim = 96;
  st = hc_config_validate(&cfg);
  printf("bad_shape %%d %%d\n", (int)st, (int)(strlen(hc_last_error_message()) > 0));
  printf("timeout_string %%s\n", hc_status_string(HC_ERR_TIMEOUT));
  return 0;
}
"""


def layout_lines():
    out = []
    for struct, fields in STRUCTS.items():
        out.append(f'  printf("size {struct} %zu\\n", sizeof({struct}));')
        for f in fields:
            out.append(f'  printf("offset {struct}.{f} %zu\\n", offsetof({struct}, {f}));')
    return "\n".join(out)


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    build.build()
    hc.load()
    d = tmp_path_factory.mktemp("c_abi")
    src = d / "abi_check.c"
    src.write_text(PROGRAM % {"layout": layout_lines(), "labels": ", ".join(map(str, LABELS_720P))})
    exe = d / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", LIB_DIR, "-lheadcast",
                    f"-Wl,-rpath,{LIB_DIR}"], check=True, capture_output=True, text=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    out = {}
    for line in run.stdout.splitlines():
        words = line.split(" ")
        if words[0] in ("size", "offset"):
            out[" ".join(words[:2])] = words[2]
        else:
            out[words[0]] = " ".join(words[1:])
    return out


def ctypes_offsets(cls):
    return {name: getattr(cls, name).offset for name, _ in cls._fields_}, C.sizeof(cls)


def test_structs_match_the_binding(c_output):
    for struct, cls in (("hc_config", hc.HcConfig), ("hc_cache_info", hc.HcCacheInfo)):
        offs, size = ctypes_offsets(cls)
        assert int(c_output[f"size {struct}"]) == size, struct
        for name, off in offs.items():
            assert int(c_output[f"offset {struct}.{name}"]) == off, (struct, name)
    dt = hc.WORK_ITEM_DTYPE
    assert int(c_output["size hc_work_item"]) == dt.itemsize
    for name in dt.names:
        assert int(c_output[f"offset hc_work_item.{name}"]) == dt.fields[name][1], name


def test_host_calls_answer_like_the_binding(c_output):
    cfg = hc.make_config(12, 128, 45, 80)
    assert int(c_output["abi"]) == hc.ABI_VERSION
    assert c_output["validate"] == "0"
    st, nbytes = c_output["cache_bytes"].split()
    assert st == "0" and int(nbytes) == hc.hc_cache_bytes(cfg, LABELS_720P)
    info = hc.hc_cache_plan_info(cfg, LABELS_720P)
    st, n_items, span = c_output["plan_info"].split()
    assert st == "0" and int(n_items) == info["n_work_items"] and int(span) == info["planned_span"]
    assert c_output["plan_count"].split() == ["0", str(info["n_work_items"])]
    assert c_output["plan_items"] == "0"
    items = hc.hc_cache_plan_items(cfg, LABELS_720P)
    w = items[0]
    assert [int(x) for x in c_output["item0"].split()] == [int(w["head"]), int(w["kind"]), int(w["q0"]), int(w["nq"]),
                                                          int(w["k_row0"]), int(w["k_len"]), int(w["cta"])]
    assert int(c_output["item_last_cta"]) == int(items[-1]["cta"])
    assert c_output["bad_shape"].split() == [str(2), "1"]      # HC_ERR_SHAPE, with a message
    assert c_output["timeout_string"] == "device-side wait expired"
