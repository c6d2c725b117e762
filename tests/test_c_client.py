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


# A C program that runs the whole decode step through the C ABI on device buffers it
# allocates itself: the inputs come from raw files, the workspace is sized with the
# contract helper dec_decode_workspace_bytes, and the results go back to files that the
# test compares with the fp64 oracle.
C_STEP_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "decattn.h"

static void *load(const char *dir, const char *name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) { fprintf(stderr, "missing %s\n", path); exit(3); }
  void *h = malloc(bytes ? bytes : 1);
  if (fread(h, 1, bytes, f) != bytes) { fprintf(stderr, "short %s\n", path); exit(3); }
  fclose(f);
  void *d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) exit(4);
  if (cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) exit(4);
  free(h);
  return d;
}

static void save(const char *dir, const char *name, const void *d, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  void *h = malloc(bytes ? bytes : 1);
  if (cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) exit(5);
  FILE *f = fopen(path, "wb");
  fwrite(h, 1, bytes, f);
  fclose(f);
  free(h);
}

int main(int argc, char **argv) {
  if (argc != 13) return 2;
  const char *dir = argv[1];
  int B = atoi(argv[2]), hidden = atoi(argv[3]), Hq = atoi(argv[4]), Hkv = atoi(argv[5]);
  int D = atoi(argv[6]), T = atoi(argv[7]), max_len = atoi(argv[8]);
  float theta = (float)atof(argv[9]);
  dec_rope_layout layout = atoi(argv[10]) ? DEC_ROPE_INTERLEAVED : DEC_ROPE_NEOX;
  int qk_norm = atoi(argv[11]);
  float eps = (float)atof(argv[12]);
  size_t act = (size_t)B * hidden * 2, qb = (size_t)B * Hq * D * 2, kvb = (size_t)B * Hkv * D * 2;
  size_t cb = (size_t)B * Hkv * T * D * 2;
  void *x = load(dir, "x.bin", act), *r = load(dir, "residual.bin", act);
  void *w = load(dir, "norm_w.bin", (size_t)hidden * 2), *q = load(dir, "q.bin", qb);
  void *kn = load(dir, "k_new.bin", kvb), *vn = load(dir, "v_new.bin", kvb);
  void *qn = qk_norm ? load(dir, "q_norm_w.bin", (size_t)D * 2) : NULL;
  void *knw = qk_norm ? load(dir, "k_norm_w.bin", (size_t)D * 2) : NULL;
  void *kc = load(dir, "k_cache.bin", cb), *vc = load(dir, "v_cache.bin", cb);
  void *pos = load(dir, "pos.bin", (size_t)B * 4), *lens = load(dir, "lens.bin", (size_t)B * 4);
  void *y = NULL, *out = NULL, *ws = NULL;
  size_t wsb = dec_decode_workspace_bytes(B, Hq, D, 0);
  if (wsb == 0 || cudaMalloc(&y, act) != cudaSuccess || cudaMalloc(&out, qb) != cudaSuccess ||
      cudaMalloc(&ws, wsb) != cudaSuccess || cudaMemset(ws, 0, wsb) != cudaSuccess)
    return 4;
  cudaStream_t s;
  if (cudaStreamCreate(&s) != cudaSuccess) return 4;
  dec_status st = dec_decode_step(x, r, w, y, hidden, eps, q, kn, vn, qn, knw, kc, vc, pos, lens,
                                  out, B, Hq, Hkv, D, T, max_len, theta, layout, NULL, 0.f, 0, 0,
                                  ws, wsb, (dec_stream_t)s);
  if (st != DEC_OK) { printf("status %d %s\n", (int)st, dec_last_error()); return 1; }
  if (cudaStreamSynchronize(s) != cudaSuccess) return 6;
  unsigned err = 0;
  if (cudaMemcpy(&err, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return 6;
  save(dir, "y.out", y, act);
  save(dir, "residual.out", r, act);
  save(dir, "q.out", q, qb);
  save(dir, "out.out", out, qb);
  save(dir, "k_cache.out", kc, cb);
  save(dir, "v_cache.out", vc, cb);
  printf("ok %d %u %d\n", (int)st, err,
         dec_decode_step_launches(B, Hq, Hkv, D, max_len, 0));
  return 0;
}
"""


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "serving_small"])
def test_plain_c_client_runs_the_decode_step(tmp_path, name):
    import numpy as np
    import torch

    import workloads as W
    from oracle import decode_ref as O
    from tol import check_float, check_ulp

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    cfg = W.TINY if name == "tiny" else W.small_variant(W.SERVING_MIX, B=6, max_len=1300)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "step.c"
    src.write_text(C_STEP_SOURCE)
    exe = tmp_path / "step"
    libdir = os.path.dirname(dsa.LIB_PATH)
    cudalib = next((p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.isdir(p)), os.path.join(cuda, "lib64"))
    subprocess.run(["gcc", "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(cuda, "include"), str(src), "-o", str(exe), "-L", libdir,
                    "-ldecattn", "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}",
                    f"-Wl,-rpath,{cudalib}"], check=True, capture_output=True, timeout=120)
    inp = W.make_inputs(cfg)
    names = ["x", "residual", "norm_w", "q", "k_new", "v_new", "k_cache", "v_cache", "pos", "lens"]
    if cfg.qk_norm:
        names += ["q_norm_w", "k_norm_w"]
    for k in names:
        t = inp[k].contiguous()
        raw = t.view(torch.int16) if t.dtype == torch.bfloat16 else t
        (tmp_path / f"{k}.bin").write_bytes(raw.numpy().tobytes())
    lens = inp["lens"].numpy()
    max_len = int(lens.max())
    r = subprocess.run([str(exe), str(tmp_path), str(cfg.B), str(cfg.hidden), str(cfg.Hq),
                        str(cfg.Hkv), str(cfg.D), str(inp["t_cap"]), str(max_len),
                        repr(float(cfg.theta)), "1" if cfg.layout == "interleaved" else "0",
                        "1" if cfg.qk_norm else "0", repr(float(cfg.eps))],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    word, st, err, launches = r.stdout.split()
    assert word == "ok" and int(st) == 0 and int(err) == 0
    assert int(launches) == dsa.decode_step_launches(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, max_len)

    def back(k, like):
        a = np.frombuffer((tmp_path / f"{k}.out").read_bytes(), dtype=np.int16).reshape(like.shape)
        return torch.from_numpy(a.copy()).view(torch.bfloat16).double().numpy()

    f64 = lambda t: t.double().numpy()
    y_ref, s_ref = O.rmsnorm_residual(f64(inp["x"]), f64(inp["residual"]), f64(inp["norm_w"]),
                                      cfg.eps)
    check_float(back("y", inp["x"]), y_ref, "C client y")
    check_ulp(back("residual", inp["x"]), s_ref, "C client residual")
    qn = None if inp["q_norm_w"] is None else f64(inp["q_norm_w"])
    kn = None if inp["k_norm_w"] is None else f64(inp["k_norm_w"])
    pos = inp["pos"].numpy()
    q_ref, kc_ref, vc_ref = O.qknorm_rope_kv_append(
        f64(inp["q"]), f64(inp["k_new"]), f64(inp["v_new"]), qn, kn, f64(inp["k_cache"]),
        f64(inp["v_cache"]), pos, cfg.theta, cfg.layout, cfg.eps)
    q_gpu = back("q", inp["q"])
    check_float(q_gpu, q_ref, "C client q")
    kc, vc = back("k_cache", inp["k_cache"]), back("v_cache", inp["v_cache"])
    for b in range(cfg.B):
        check_ulp(kc[b, :, pos[b]], kc_ref[b, :, pos[b]], "C client K slot")
        assert np.array_equal(vc[b, :, pos[b]], vc_ref[b, :, pos[b]])
    out_ref = O.gqa_decode_attention(q_gpu, kc, vc, lens)
    check_float(back("out", inp["q"]), out_ref, "C client out")
