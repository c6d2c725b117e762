"""The C ABI from a plain C program (no Python in between): compiled with gcc against
include/decattn.h, linked to the library, run on the CPU with host-only calls."""
import os
import shutil
import subprocess

import pytest

import decode_step_attention_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include "decattn.h"

int main(void) {
  double t[64];
  float scale = 0.f;
  dec_status st = dec_rope_inv_freq(128, 500000.f, DEC_ROPE_SCALE_NTK, 4.f, t);
  if (st != DEC_OK) { printf("err %d %s\n", (int)st, dec_status_string(st)); return 1; }
  if (dec_rope_yarn_softmax_scale(128, 8.f, &scale) != DEC_OK) return 2;
  /* a bad head_dim is refused with a status and a message, nothing else */
  st = dec_rope_inv_freq(96, 1e4f, DEC_ROPE_SCALE_NONE, 1.f, t);
  printf("%d %.17g %.17g %.9g %d %s %zu\n", dec_version(), t[0], t[63], (double)scale,
         (int)st, dec_status_string(st), dec_attn_workspace_bytes(4, 32, 8, 128, 4096, 152));
  return 0;
}
"""


def test_plain_c_client(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    if not os.path.exists(dsa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    src = tmp_path / "client.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "client"
    libdir = os.path.dirname(dsa.LIB_PATH)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    str(src), "-o", str(exe), "-L", libdir, "-ldecattn", f"-Wl,-rpath,{libdir}"],
                   check=True, capture_output=True, timeout=120)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    ver, f0, f63, scale, st, msg, ws = r.stdout.split(maxsplit=6)
    table = dsa.rope_inv_freq(128, 5e5, "ntk", 4.0)
    assert int(ver) == dsa.lib().dec_version()
    assert float(f0) == float(table[0]) and float(f63) == float(table[63])
    assert abs(float(scale) - dsa.yarn_softmax_scale(128, 8.0)) <= 1e-7
    assert int(st) == 2 and "unsupported" in msg.lower()
    assert int(ws.split()[-1]) == dsa.lib().dec_attn_workspace_bytes(4, 32, 8, 128, 4096, 152)
