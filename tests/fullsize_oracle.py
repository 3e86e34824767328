"""Oracle comparison of many heads at once, spread over host processes.

Test infrastructure (imports the oracle): the full-size parity tests hand the
CUDA path's outputs to this module, which checks every requested (b, h) head
element by element against the float64 oracle on the same seeded inputs.

The inputs' storage form and the outputs are written once to a temporary
directory as .npy files; worker processes (started with the ``spawn`` method,
each with one BLAS thread) map them read-only, run ``oracle.attention``'s
``backward_head`` (which also returns the forward's O and LSE) on their share
of the heads and send back the worst error and mismatch count per tensor.
"""

import multiprocessing as mp
import os
import tempfile
from concurrent.futures import ProcessPoolExecutor

import numpy as np

from exact_attention_fwd_gb300.inputs import bf16_bits_to_f64, f32_to_bf16_bits

_GRADS = ("dq", "dk", "dv")


def _as_f64(arr, kind):
    return bf16_bits_to_f64(arr) if kind == "bf16" else np.asarray(arr, dtype=np.float64)


def _round_bf16(x):
    """float64 -> nearest bf16 (through float32), back as float64."""
    return bf16_bits_to_f64(f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _worker(job):
    from oracle import attention as A
    from oracle import checker
    d = job["dir"]
    kinds = job["kinds"]
    arr = {n: np.load(os.path.join(d, n + ".npy"), mmap_mode="r") for n in kinds}
    worst = {}
    fails = []
    for b, h in job["heads"]:
        qh, kh, vh, dh = (_as_f64(arr[t][b, :, h, :], job["in_kind"]) for t in ("q", "k", "v", "do"))
        g = A.backward_head(qh, kh, vh, dh, job["scale"], job["causal"])
        checks = [("o", _as_f64(arr["o"][b, :, h, :], kinds["o"]), g["O"], job["tol"]["o"]),
                  ("lse", np.asarray(arr["lse"][b, h], dtype=np.float64), g["lse"],
                   job["tol"]["lse"])]
        for name in _GRADS:
            if name in arr:
                checks.append((name, _as_f64(arr[name][b, :, h, :], kinds[name]), g[name],
                               job["tol"]["grad"]))
        for name in job.get("report", ()):
            # bf16-stored gradients: error against the bf16-rounded oracle value
            got = _as_f64(arr[name][b, :, h, :], kinds[name])
            e = float(np.max(np.abs(got - _round_bf16(g[name[:-5]]))))
            worst[name] = max(worst.get(name, 0.0), e)
            worst[name + "_vs_f64"] = max(worst.get(name + "_vs_f64", 0.0),
                                         float(np.max(np.abs(got - g[name[:-5]]))))
        for name, got, ref, tol in checks:
            ok, e, n = checker.check(got, ref, tol)
            worst[name] = max(worst.get(name, 0.0), e)
            if not ok:
                fails.append(f"{name} head {(b, h)}: max err {e:.3e}, {n} mismatches")
        worst["max_abs_ref"] = max(worst.get("max_abs_ref", 0.0),
                                   *(float(np.max(np.abs(g[n]))) for n in _GRADS))
    return worst, fails


def workers_for(bytes_per_worker, cap=16):
    """Worker count that fits the host: at most `cap`, the core count, and
    what MemAvailable (Linux) holds at `bytes_per_worker` each, with a
    quarter kept free."""
    n = min(cap, os.cpu_count() or 1)
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    avail = int(ln.split()[1]) * 1024
                    n = min(n, max(1, int(0.75 * avail // bytes_per_worker)))
                    break
    except OSError:
        pass
    return n


def _save(d, name, a):
    np.save(os.path.join(d, name + ".npy"), np.ascontiguousarray(a))


def check_heads(inp, outputs, heads, scale, causal, tol, workers=None, report=()):
    """Compare the given heads of `outputs` with the oracle.

    inp: exact_attention_fwd_gb300.inputs.Inputs (bf16 or f32 storage).
    outputs: dict name -> (numpy array, kind) with kind "bf16" (uint16 bit
    patterns) or "f32"; names o, lse and any of dq, dk, dv; extra names in
    `report` (e.g. "dq_bf16") are compared with the bf16-rounded oracle value
    of the gradient their name starts with, without a tolerance.
    Returns (worst error per tensor, list of failure messages).
    """
    workers = workers or min(16, os.cpu_count() or 1)
    heads = list(heads)
    in_kind = "bf16" if inp.dtype == "bf16" else "f32"
    with tempfile.TemporaryDirectory(prefix="fa_fullsize_") as d:
        kinds = {}
        for t in ("q", "k", "v", "do"):
            _save(d, t, inp.storage[t])
            kinds[t] = in_kind
        for name, (a, kind) in outputs.items():
            _save(d, name, a)
            kinds[name] = kind
        chunks = [heads[i::workers] for i in range(workers)]
        jobs = [dict(dir=d, kinds=kinds, in_kind=in_kind, heads=c, scale=scale, causal=causal,
                     tol=tol, report=tuple(report)) for c in chunks if c]
        # one BLAS thread per worker (the environment is read when numpy loads)
        saved = {v: os.environ.get(v) for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                                                "MKL_NUM_THREADS")}
        for v in saved:
            os.environ[v] = "1"
        try:
            with ProcessPoolExecutor(max_workers=len(jobs),
                                     mp_context=mp.get_context("spawn")) as ex:
                results = list(ex.map(_worker, jobs))
        finally:
            for v, val in saved.items():
                if val is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = val
    worst, fails = {}, []
    for w, f in results:
        for k, e in w.items():
            worst[k] = max(worst.get(k, 0.0), e)
        fails.extend(f)
    return worst, fails
