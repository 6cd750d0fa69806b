"""Writes the stored expected values under tests/golden/ using only the oracle.

batch_split_ticket.json: the ticket shape of the page "ROCm/rocm-libraries
PR #11188" ("Motivation": nn.Conv2d(96, 64, 1) on a [64, 96, 512, 512] fp32
input; "Test Plan": batch sizes n = 43..192). The "~4GB" per-dispatch limit is
read as 2^32 bytes of X per dispatch, so max_n = floor(2^32 / bytes per sample).
Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def main():
    orc = oracle.get()
    bytes_per_sample = 96 * 512 * 512 * 4
    max_n = (2 ** 32) // bytes_per_sample
    out = {
        "source": "ROCm/rocm-libraries PR #11188, 'Motivation' (ticket shape) and 'Test Plan' (n = 43..192)",
        "reading": "limit = 2^32 bytes of X per dispatch; max_n = floor(limit / bytes_per_sample)",
        "bytes_per_sample": bytes_per_sample,
        "max_n": max_n,
        "split_count": {str(n): orc.batch_split_count(n, max_n) for n in list(range(1, 43)) + list(range(43, 193))},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "batch_split_ticket.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
