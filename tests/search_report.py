"""Record of the alpha-index decisions the GPU search tests compare with the oracle.

Every comparison adds one entry; a GPU pick other than the oracle's argmin is only accepted on
a near-tie of the oracle's own errors, and each such acceptance is listed in pytest's terminal
summary (tests/conftest.py), so a run shows how many there were (the target is none).
"""

COMPARED = []     # (label, gpu index, oracle index, relative oracle gap best -> runner-up)
ACCEPTED = []     # (label, gpu index, oracle index, relative gap E(gpu) / E(oracle) - 1, allowed)


def compared(label, b_gpu, b_oracle, runner_gap):
    COMPARED.append((label, int(b_gpu), int(b_oracle), float(runner_gap)))


def accepted(label, b_gpu, b_oracle, rel_gap, allowed):
    ACCEPTED.append((label, int(b_gpu), int(b_oracle), float(rel_gap), float(allowed)))


def summary_lines():
    if not COMPARED:
        return []
    close = sum(1 for c in COMPARED if c[3] < 1e-4)
    out = [f"alpha index vs oracle: {len(COMPARED)} searches compared, "
           f"{len(COMPARED) - len(ACCEPTED)} exact, {len(ACCEPTED)} near-ties accepted "
           f"(oracle best and runner-up within 1e-4 relative in {close})"]
    for label, b, r, gap, allowed in ACCEPTED:
        out.append(f"  near-tie {label}: gpu alpha index {b}, oracle {r}, "
                   f"E_oracle({b}) / E_oracle({r}) - 1 = {gap:.3e} (allowed {allowed:.3e})")
    return out
