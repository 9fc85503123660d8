"""The boundary from C: a plain C99 program includes include/gbconv.h, links the built library and
calls the entry points that need no GPU (output shape, family, plan, host staging size, status
strings, argument checks).  Its printout is compared with the Python binding and the oracle, so the
header's types and the exported symbols agree for a C caller, not only through ctypes.
"""
import os
import shutil
import subprocess

import pytest

from tests.helpers import lib_desc, oracle_conv, shape_kw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "gbconv.h"

int main(void) {
  gbconv_desc d;
  memset(&d, 0, sizeof d);
  d.spatial_dims = 2;
  d.layout = GBCONV_NHWC;
  d.wlayout = GBCONV_W_OHWI;
  d.dtype = GBCONV_BF16;
  d.n = 32; d.c_in = 64; d.c_out = 64; d.groups = 1;
  d.in[0] = 56; d.in[1] = 56; d.k[0] = 3; d.k[1] = 3;
  d.stride[0] = 2; d.stride[1] = 2; d.pad[0] = 1; d.pad[1] = 1; d.dil[0] = 1; d.dil[1] = 1;
  int64_t out[3] = {0, 0, 0};
  if (gbconv_out_shape(&d, out) != GBCONV_OK) return 10;
  int32_t fam_fwd = -1, fam_dgrad = -1, fam_wgrad = -1;
  if (gbconv_select(&d, GBCONV_OP_FWD, &fam_fwd) != GBCONV_OK) return 11;
  if (gbconv_select(&d, GBCONV_OP_BWD_DATA, &fam_dgrad) != GBCONV_OK) return 12;
  if (gbconv_select(&d, GBCONV_OP_BWD_FILTER, &fam_wgrad) != GBCONV_OK) return 13;
  char plan[256];
  if (gbconv_describe(&d, GBCONV_OP_FWD, plan, (int64_t)sizeof plan) != GBCONV_OK) return 14;
  int64_t staging = 0, workspace = 0;
  if (gbconv_host_staging_bytes(&d, GBCONV_OP_FWD, 1, &staging) != GBCONV_OK) return 15;
  if (gbconv_bwd_filter_workspace(&d, &workspace) != GBCONV_OK) return 16;
  /* argument errors come back before anything touches a device */
  if (gbconv_fwd(&d, NULL, NULL, NULL, NULL, NULL) != GBCONV_EINVAL) return 17;
  gbconv_desc bad = d;
  bad.k[0] = 200;
  if (gbconv_out_shape(&bad, out) != GBCONV_EINVAL) return 18;
  printf("out %lld %lld %lld\n", (long long)out[0], (long long)out[1], (long long)out[2]);
  printf("families %d %d %d\n", (int)fam_fwd, (int)fam_dgrad, (int)fam_wgrad);
  printf("plan %s\n", plan);
  printf("staging %lld\n", (long long)staging);
  printf("workspace %lld\n", (long long)workspace);
  printf("status %s|%s\n", gbconv_status_string(GBCONV_OK), gbconv_status_string(GBCONV_ETIMEOUT));
  return 0;
}
"""


@pytest.fixture(scope="module")
def gb():
    import __graft_entry__
    __graft_entry__.build()
    import convolution_conv_fwd_gb300 as gb
    return gb


def test_c_program_calls_the_library(gb, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "client"
    libdir = os.path.dirname(gb.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir,
                    "-lgbconv", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True, capture_output=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    lines = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())
    kw = shape_kw(n=32, in_size=(56, 56), c_in=64, c_out=64, stride=(2, 2))
    c = oracle_conv(kw)
    assert lines["out"] == "%d %d 1" % (c.y_shape()[1], c.y_shape()[2])  # NHWC: (N, OH, OW, C)
    d = lib_desc(gb, kw)
    fams = [int(v) for v in lines["families"].split()]
    assert [gb.KERNELS[f] for f in fams] == [gb.gbconv_select(d, op) for op in (0, 1, 2)]
    assert lines["plan"] == gb.gbconv_describe(d, 0)
    assert int(lines["staging"]) == gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_FWD, True)
    assert int(lines["workspace"]) == gb.gbconv_bwd_filter_workspace(d)
    assert lines["status"] == "%s|%s" % (gb.status_string(0), gb.status_string(4))
