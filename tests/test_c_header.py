"""include/gdn.h from plain C: a C99 program includes the header with every
warning an error, links against libgdn.so and makes the host-only calls (status
strings, size queries, the scan plan, the slot-index check, argument checks that
return before any launch).  No GPU is needed."""
import os
import shutil
import subprocess
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "chunked_gated_delta_06_gb300")

PROGRAM = textwrap.dedent(r"""
    #include <stddef.h>
    #include <stdio.h>
    #include <string.h>
    #include "gdn.h"

    int main(void) {
        int32_t cu[4] = {0, 1, 64, 200};
        gdn_problem p;
        memset(&p, 0, sizeof p);
        p.num_seqs = 3; p.total_tokens = 200; p.num_k_heads = 2; p.num_v_heads = 4;
        p.head_dim_k = 128; p.head_dim_v = 128; p.scale = 0.0f;
        p.cu_seqlens_host = cu;
        p.cu_seqlens_dev = (const int32_t *)(uintptr_t)0x1000;   /* never read by a host call */
        if (strncmp(gdn_status_string(GDN_ERR_UNSUPPORTED), "GDN_ERR_UNSUPPORTED", 19)) return 1;
        if (gdn_chunk_saved_bytes(&p) == 0 || gdn_chunk_workspace_bytes(&p, 0) == 0) return 2;
        int32_t seg_len = -1, nseg = -1;
        if (gdn_chunk_scan_plan(&p, &seg_len, &nseg) != GDN_OK || nseg != 1) return 3;
        int32_t idx[5] = {3, 0, -1, 3, 2}, bad = -2;
        if (gdn_check_indices(idx, 5, 8, &bad) != GDN_ERR_INVALID_ARG || bad != 3) return 4;
        /* argument checks return before any launch */
        if (gdn_chunk_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL)
            != GDN_ERR_INVALID_ARG) return 5;
        p.head_dim_v = 64;
        if (gdn_chunk_saved_bytes(&p) != 0) return 6;
        /* a zeroed struct is the library's plan; -1 never splits; -2 is rejected */
        p.head_dim_v = 128;
        p.scan_segment_chunks = -2;
        if (gdn_chunk_scan_plan(&p, &seg_len, &nseg) != GDN_ERR_INVALID_ARG) return 7;
        p.scan_segment_chunks = -1;
        if (gdn_chunk_scan_plan(&p, &seg_len, &nseg) != GDN_OK || seg_len != 0) return 8;
        p.device_status = (int32_t *)(uintptr_t)0x1002;   /* misaligned: rejected */
        if (gdn_chunk_workspace_bytes(&p, 0) != 0) return 9;
        printf("ok %zu %zu %zu\n", sizeof(gdn_problem), offsetof(gdn_problem, device_status),
               offsetof(gdn_problem, scan_segment_chunks));
        return 0;
    }
""")


def test_header_compiles_as_c99_and_host_calls_work(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from chunked_gated_delta_06_gb300 import build
    build.build()
    src = tmp_path / "use_gdn.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_gdn"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", PKG, "-lgdn", "-Wl,-rpath," + PKG, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    # the same layout the ctypes binding declares
    assert out.stdout.strip() == "ok 72 56 64"
