"""include/hc.h is a plain C interface: a C99 program (gcc -std=c99 -pedantic
-Werror) and a C++11 program include it, link libhc.so and call its host
helpers, which need no GPU.  Their answers are compared with what the
pages fix (Ring AllReduce 2(P-1) steps, RHD 2 ceil(log2 P)) and with the
library's own Python binding."""
import os
import shutil
import subprocess

import pytest

from collective_communication_algorithms_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "hc.h"

int main(void) {
    hc_stats_t st;
    size_t off = 0, len = 0;
    hc_algo_t algo = HC_ALGO_RING;
    double t = 0.0;
    int k;
    memset(&st, 0, sizeof st);
    st.struct_size = sizeof st;
    printf("version %d\n", hc_version());
    printf("status %s\n", hc_status_string(HC_ERR_INVALID_ARG));
    if (hc_schedule_stats(HC_ALGO_RING, HC_COLL_ALLREDUCE, 8, 1, 4096, HC_FLOAT32, 0, &st, NULL) != HC_OK)
        return 2;
    printf("ring_steps %d\n", st.steps_per_loop);
    if (hc_schedule_stats(HC_ALGO_RHD, HC_COLL_ALLREDUCE, 5, 1, 4096, HC_INT32, 0, &st, NULL) != HC_OK)
        return 3;
    printf("rhd5_steps %d\n", st.steps_per_loop);
    printf("segments %d\n", hc_num_segments(HC_ALGO_RING, HC_COLL_REDUCE_SCATTER, 3));
    for (k = 0; k < 3; k++) {
        if (hc_segment_range(HC_ALGO_RING, HC_COLL_REDUCE_SCATTER, 3, 1001, HC_FLOAT32, k, &off, &len) != HC_OK)
            return 4;
        printf("seg %d %zu %zu\n", k, off, len);
    }
    if (hc_select_algo(HC_COLL_ALLREDUCE, 8, 1, 1024, HC_FLOAT32, HC_MODE_STEP, &algo, &t) != HC_OK)
        return 5;
    printf("select %d\n", (int)algo);
    /* rejected before any launch: P = 0 */
    printf("bad %d\n", (int)hc_allreduce(NULL, NULL, 0, 16, HC_FLOAT32, HC_SUM, HC_ALGO_RING, NULL, NULL));
    return 0;
}
"""


def lib_dir():
    from collective_communication_algorithms_gb300 import build
    build.build()
    return os.path.dirname(B.LIB_PATH)


@pytest.mark.parametrize("compiler,std,suffix", [("gcc", "-std=c99", ".c"), ("g++", "-std=c++11", ".cpp")])
def test_header_is_plain_c_and_links(tmp_path, compiler, std, suffix):
    if shutil.which(compiler) is None:
        pytest.skip(compiler + " not found")
    d = lib_dir()
    src = tmp_path / ("consumer" + suffix)
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    cmd = [compiler, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", INCLUDE, str(src),
           "-L", d, "-lhc", "-Wl,-rpath," + d, "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(line.split(" ", 1) for line in out if line)
    assert int(got["version"]) == B.hc_version()
    assert got["status"] == B.status_string(1)
    assert int(got["ring_steps"]) == 2 * (8 - 1)
    assert int(got["rhd5_steps"]) == 2 * 3  # 2 ceil(log2 5)
    assert int(got["segments"]) == 3
    for k in range(3):
        off, ln = B.hc_segment_range("ring", "reducescatter", 3, 1001, "float32", k)
        assert [int(x) for x in [l for l in out if l.startswith("seg %d " % k)][0].split()[2:]] == [off, ln]
    assert int(got["select"]) == B.ALGOS[B.hc_select_algo("allreduce", 8, 1024, "float32", "step", 1)[0]]
    assert int(got["bad"]) == 1  # HC_ERR_INVALID_ARG
