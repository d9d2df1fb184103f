"""The boundary from plain C: a C99 program that includes only
include/sfa_grad.h and links libsfa.so calls the host-side entry points
(workspace sizes, plan queries, validation, status strings) and must get what
the Python binding gets.  No GPU call is made."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "sfa_grad.h"

#define FAKE ((void*)(size_t)16) /* never dereferenced: the call is rejected first */

static sfa_params mla(int det) {
  sfa_params p;
  memset(&p, 0, sizeof(p));
  p.layout = SFA_LAYOUT_BSND;
  p.dtype = SFA_DTYPE_BF16;
  p.B = 1; p.S1 = 4096; p.S2 = 4096;
  p.N1 = 128; p.N2 = 1; p.D = 512; p.Dr = 64; p.K = 2048;
  p.scale = 0.041666666666666664;
  p.sparse_block_size = 1;
  p.sparse_mode = 0;
  p.deterministic = det;
  return p;
}

int main(void) {
  for (int det = 0; det <= 1; ++det) {
    sfa_params p = mla(det);
    size_t ws = 0, hws = 0;
    int64_t chunk = 0, launches = 0;
    int32_t n = 0;
    if (sfa_grad_workspace_size(&p, &ws) != SFA_OK) return 2;
    if (sfa_grad_host_workspace_size(&p, &hws) != SFA_OK) return 3;
    if (sfa_grad_plan_info(&p, &chunk, &launches) != SFA_OK) return 4;
    if (sfa_grad_plan_names(&p, NULL, 0, &n) != SFA_OK || n != launches) return 5;
    const char* names[64];
    if (n > 64 || sfa_grad_plan_names(&p, names, n, &n) != SFA_OK) return 6;
    printf("det=%d ws=%zu host_ws=%zu chunk=%lld launches=%lld names=", det, ws, hws, (long long)chunk,
           (long long)launches);
    for (int i = 0; i < n; ++i) printf("%s%s", i ? "," : "", names[i]);
    printf("\n");
  }
  /* validation codes, before any device work */
  sfa_params bad = mla(0);
  bad.N2 = 2;
  size_t ws = 0;
  printf("n2=%d\n", (int)sfa_grad_workspace_size(&bad, &ws));
  printf("null=%d\n", (int)sfa_grad_workspace_size(NULL, &ws));
  sfa_params p = mla(0);
  printf("short_ws=%d\n", (int)sfa_grad(&p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL, FAKE,
                                        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, NULL));
  printf("status=%s\n", sfa_status_string(SFA_ERR_SHAPE));
  return 0;
}
"""


@pytest.fixture(scope="module")
def built():
    from sfa_grad_gb300.build import build
    build()
    import sfa_grad_gb300 as m
    m.lib()
    return m


def test_c_program_calls_the_abi(built, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "abi"
    libdir = os.path.join(ROOT, "sfa_grad_gb300")
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lsfa", f"-Wl,-rpath,{libdir}"], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    out = dict(line.split("=", 1) for line in r.stdout.splitlines() if "=" in line and not line.startswith("det="))
    assert int(out["n2"]) == built.SFA_ERR_SHAPE
    assert int(out["null"]) == built.SFA_ERR_NULLPTR
    assert int(out["short_ws"]) == built.SFA_ERR_PARAM_INVALID
    assert out["status"].startswith("SFA_ERR_SHAPE")
    # the same plan as the Python binding reports
    rows = [line for line in r.stdout.splitlines() if line.startswith("det=")]
    assert len(rows) == 2
    for det, line in enumerate(rows):
        f = dict(kv.split("=", 1) for kv in line.split(" "))
        p = built.SfaParams()
        for k, v in dict(layout=0, dtype=0, B=1, S1=4096, S2=4096, T1=0, T2=0, N1=128, N2=1, D=512, Dr=64, K=2048,
                         scale=1 / 24, sparse_block_size=1, sparse_mode=0, deterministic=det).items():
            setattr(p, k, v)
        assert int(f["ws"]) == built.grad_workspace_size(p)
        assert int(f["host_ws"]) == built.grad_host_workspace_size(p)
        chunk, launches = built.plan_info(p)
        assert int(f["chunk"]) == chunk and int(f["launches"]) == launches
        assert f["names"].split(",") == built.plan_names(p)
