"""Summarise an ncu launch list (``--metrics gpu__time_duration.sum --csv``) per kernel.

    python -m decoder_only_transformer_gpt_gb300.ncu_summary launches.csv [--skip N] [--take N] [--steps S]
                                                                          [--layers L]

Prints a markdown table: kernel, launches, total time, time per step and share.
--skip drops the first N launches (warm-up), --take keeps the next N (0 = all),
--steps divides totals into per-step figures. With --layers L the launches are
also labelled by their step of the pre-norm bf16 forward pass of an L-block
model (embed, then per block c_attn, attention, c_proj, ln_2, c_fc, mlp c_proj,
next LayerNorm, then head, CE combine, mean) and a second table is printed per
step kind; --skip must then land on a step boundary.
"""
import argparse
import collections
import csv
import re

_SCALE = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3}

BLOCK_STEPS = ["c_attn", "attention", "c_proj", "ln_mid", "c_fc", "mlp_proj", "ln_out"]


def load(path):
    rows = list(csv.reader(open(path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Value" in r)
    h = rows[hi]
    ki, vi, ui, ii = h.index("Kernel Name"), h.index("Metric Value"), h.index("Metric Unit"), h.index("ID")
    out = []
    for r in rows[hi + 1:]:
        if len(r) <= max(ki, vi, ui, ii):
            continue
        us = float(r[vi].replace(",", "")) * _SCALE[r[ui]]
        out.append((int(r[ii]), r[ki], us))
    out.sort()
    return out


def short(name: str) -> str:
    name = re.sub(r"\(CUtensorMap_st.*|\(const .*|\(int.*", "", name)
    return name.replace("gptgb::<unnamed>::", "").replace("void ", "")


def step_names(layers: int):
    return ["embed"] + BLOCK_STEPS * layers + ["head", "ce_combine", "mean"]


def _table(agg, steps, first_col):
    total = sum(a[1] for a in agg.values())
    lines = [f"| {first_col} | launches | total us | us / step | share |", "|---|---:|---:|---:|---:|"]
    for k, (n, t) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        lines.append(f"| `{k}` | {n} | {t:.1f} | {t / steps:.1f} | {100 * t / total:.1f}% |")
    lines.append(f"| **all** | {sum(a[0] for a in agg.values())} | {total:.1f} | {total / steps:.1f} | 100% |")
    return "\n".join(lines)


def summarise(launches, skip=0, take=0, steps=1, layers=0):
    sel = launches[skip:skip + take] if take else launches[skip:]
    agg = collections.OrderedDict()
    for _, k, us in sel:
        a = agg.setdefault(short(k), [0, 0.0])
        a[0] += 1
        a[1] += us
    out = _table(agg, steps, "kernel")
    if layers:
        names = step_names(layers)
        by_step = collections.OrderedDict()
        for i, (_, _, us) in enumerate(sel):
            a = by_step.setdefault(names[i % len(names)], [0, 0.0])
            a[0] += 1
            a[1] += us
        out += "\n\n" + _table(by_step, steps, "step")
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("csv")
    ap.add_argument("--skip", type=int, default=0)
    ap.add_argument("--take", type=int, default=0)
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--layers", type=int, default=0)
    a = ap.parse_args()
    print(summarise(load(a.csv), a.skip, a.take, a.steps, a.layers))
