"""Stand-in replica for the multi-rank bench test (CPU, gloo backend): bench.py's own
rank flow (Ranks, replica_rate, WallClock) around a host step whose length depends on
the rank, so that the whole-job rate must use the slowest rank's time.  Started by
torch.distributed.run through bench.launch_replicas; rank 0 prints one JSON line."""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

STEPS = 5


def main():
    ranks = bench.Ranks("gloo")
    delay = 0.02 * (1 + ranks.rank)   # rank 1 takes twice as long per step
    rate, elapsed = bench.replica_rate(ranks, lambda: time.sleep(delay), STEPS, 100.0,
                                       bench.WallClock())
    if ranks.rank == 0:
        print(json.dumps({"n_gpus": ranks.ws, "value": rate, "elapsed_s": elapsed,
                          "steps": STEPS, "delay_s": delay}), flush=True)
    ranks.close()


if __name__ == "__main__":
    main()
