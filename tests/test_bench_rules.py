"""Host-side rules of the benchmark's decode lines, on the CPU.

* The kernels a decode layer launches per step (the `gpu_launches` claim)
  follow the library's plan: a row's 64-key tiles split over
  min(SMs // rows, tiles) items, items of at most 4 tiles expanding the cache
  rows themselves, longer ones reading rows gathered by one more kernel.  On
  a 148-SM B300 the ncu launch lists of these workloads show 6 kernels per
  step for the 4 x 1M hybrid pair (CSA: append, scores, top-k, attention;
  HCA: append, attention), 5 for 32 x 128K CSA (with the row gather) and 3
  for 16 x 1M HCA (append, row gather, attention).
* The recorded DRAM traffic of the 4 x 1M step cannot be below its
  algorithmic bytes: the resident caches (~0.7 GB) are far larger than L2,
  so every byte the step must read comes from DRAM at least once.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def test_decode_kernels_per_step_match_the_launch_lists():
    c = wl.CONFIGS
    hybrid = [c["c5_hybrid_csa_decode_1m"], c["c5_hybrid_hca_decode_1m"]]
    assert [bench.decode_layer_kernels(x, 148) for x in hybrid] == [4, 2]
    assert bench.decode_layer_kernels(c["c3_csa_decode_128k"], 148) == 5
    assert bench.decode_layer_kernels(c["c4_hca_decode_1m"], 148) == 3


def test_decode_step_traffic_is_not_below_the_algorithmic_bytes():
    c = wl.CONFIGS
    alg = bench.decode_bytes(c["c5_hybrid_csa_decode_1m"]) + bench.decode_bytes(c["c5_hybrid_hca_decode_1m"])
    assert alg == 59693112.0
    traffic = bench.DECODE_STEP_TRAFFIC["c5_hybrid_csa_decode_1m"]
    assert alg <= traffic <= 1.2 * alg
