"""Summarise an ncu launch list (``--metrics gpu__time_duration.sum --csv``)
into per-kernel launches, total device time and share of the total."""
import collections
import csv
import re
import sys

UNIT = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3}
KERNEL = re.compile(r"(attn_\w+|rows_kernel|partition_kernel|accum_cast_kernel|zero_tail_kernel"
                    r"|\w+_kernel)(<[^>]*>)?")


def summarise(path):
    rows = list(csv.reader(open(path)))
    start = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    hdr, data = rows[start], rows[start + 1:]
    ki, mi, ui, vi = (hdr.index(c) for c in ("Kernel Name", "Metric Name", "Metric Unit",
                                             "Metric Value"))
    agg = collections.defaultdict(lambda: [0, 0.0])
    for r in data:
        if r[mi] != "gpu__time_duration.sum":
            continue
        m = KERNEL.search(r[ki])
        name = m.group(0) if m else r[ki][:60]
        agg[name][0] += 1
        agg[name][1] += float(r[vi].replace(",", "")) * UNIT[r[ui]]
    return agg


if __name__ == "__main__":
    agg = summarise(sys.argv[1])
    tot = sum(t for _, t in agg.values())
    print("| kernel | launches | total (us) | share |")
    print("|---|---:|---:|---:|")
    for k, (n, t) in sorted(agg.items(), key=lambda x: -x[1][1]):
        print(f"| `{k}` | {n} | {t:.1f} | {100 * t / tot:.2f}% |")
    print(f"| total | {sum(n for n, _ in agg.values())} | {tot:.1f} | 100% |")
