"""The C ABI from C and C++ (CPU): include/fathom.h compiles on its own as C11
and C++17, a C program links against libfathom.so, takes the address of every
declared entry point, and exercises the host-only paths (version, workspace
sizes, argument errors with their messages).  No kernel is launched."""
import os
import re
import subprocess

import pytest

from bit_plane_kv_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
HEADER = os.path.join(INC, "fathom.h")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fathom.h"

typedef void (*any_fn)(void);

int main(void) {
    any_fn fns[] = { %(fns)s };
    for (size_t i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i)
        if (!fns[i]) { printf("null entry %%zu\n", i); return 1; }
    if (!strstr(fathom_version(), "sm_103a")) { printf("version\n"); return 1; }

    fathom_shape s = {2, 4096, 128, 4, 512, 4, 32, 0};
    size_t ws = fathom_workspace_size(&s, FATHOM_WS_SCAN_TOPK);
    size_t wa = fathom_workspace_size(&s, FATHOM_WS_SPARSE_ATTN);
    if (ws == 0 || wa == 0 || (ws & 255) || (wa & 255)) { printf("workspace sizes\n"); return 1; }

    fathom_shape bad = s;
    bad.G = 3;
    if (fathom_workspace_size(&bad, FATHOM_WS_SCAN_TOPK) != 0) { printf("bad shape accepted\n"); return 1; }
    if (!strstr(fathom_last_error(), "G must")) { printf("message: %%s\n", fathom_last_error()); return 1; }

    int rc = fathom_quantize_pack(&s, NULL, FATHOM_BF16, (uint64_t *)256, (uint16_t *)256, NULL);
    if (rc != FATHOM_EINVAL || strcmp(fathom_last_error(), "keys is NULL")) { printf("null check\n"); return 1; }
    printf("ok %%zu %%zu\n", ws, wa);
    return 0;
}
"""


def declared():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(fathom_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_dir():
    return os.path.dirname(BUILD.build())


@pytest.mark.parametrize("lang,std", [("c", "-std=c11"), ("c++", "-std=c++17")])
def test_header_compiles_alone(lang, std, tmp_path):
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "fathom.h"\nint fathom_header_only_check;\n')
    cc = "gcc" if lang == "c" else "g++"
    subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INC, "-c", str(src),
                    "-o", str(tmp_path / "h.o")], check=True, capture_output=True, text=True)


def test_c_program_links_and_runs_host_paths(lib_dir, tmp_path):
    fns = ", ".join(f"(any_fn){name}" for name in declared())
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM % {"fns": fns})
    exe = tmp_path / "prog"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", INC, str(src), "-o", str(exe),
                    "-L", lib_dir, "-lfathom", f"-Wl,-rpath,{lib_dir}"], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok "), r.stdout + r.stderr
