"""Writes fidelity_report.json: the oracle's fidelity report (attention output
of the mixed BF16 / INT2 cache against all-BF16 attention, and the INT2 keys'
and values' reconstruction error) for OSCAR, Hadamard-only and unrotated INT2
on the tiny workload and the Qwen3-8B-shaped 32768-token workload, with the
workloads' own calibration sizes.  Calls only the oracle and the seeded input
generator; the numbers are a report, not a target (the pages print none for
synthetic inputs).

    python tests/golden/fidelity_report.py      # a few minutes on one host
"""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from int2_rotated_kv_gb300 import synth  # noqa: E402
from oracle import attention  # noqa: E402


def main():
    out = {}
    for w in (synth.TINY, synth.QWEN3_8B_32K):
        t0 = time.time()
        inst = synth.draw_instance(w)
        rep = attention.fidelity_report(inst, sink=w.sink, window=w.window)
        out[w.name] = {"context": int(inst.seq_lens[0]), "n_calib": w.n_calib,
                       "sink": w.sink, "window": w.window, **rep}
        print(w.name, json.dumps(rep), f"{time.time() - t0:.0f} s", flush=True)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fidelity_report.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
