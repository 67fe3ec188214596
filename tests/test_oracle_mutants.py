"""The oracle's pins must catch a planted mistake anywhere in the oracle.

Each mutant below is one plausible slip in `oracle/ss_oracle.c`: a dropped
term, a wrong divisor, a reversed order, a transposed index, an off-by-one
rule.  The test writes the mutated source to a temporary directory, compiles
it with the oracle's own flags, and runs the pin suite
(`tests/test_oracle_pins.py`) against that library through SSO_ORACLE_LIB.
At least one pin has to fail for every mutant.  The planted mistakes live
only in the temporary copies, on the CPU; every mutant keeps its reads and
writes inside the buffers the callers allocate.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "ss_oracle.c")

# (name, exact text in ss_oracle.c, replacement).  Only mutants that change
# some result are listed: reordering the reduce-scatter's loop over shards,
# for one, computes every output from the same inputs and is no mistake.
MUTANTS = [
    # bf16 rounding
    ("bf16 ties away from zero",
     "    if (dropped > half || (dropped == half && (upper & 1u))) {",
     "    if (dropped >= half) {"),
    ("bf16 NaN keeps only its upper half (low-payload NaNs become infinities)",
     "        return (uint16_t)((u >> 16) | 0x0040u);",
     "        return (uint16_t)(u >> 16);"),
    # layout
    ("FLAT_ORIG_TRUE alignment of 8 elements whatever the dtype",
     "        int64_t a = 16 / elem_bytes;",
     "        int64_t a = 8;"),
    ("FLAT_ORIG_FALSE chunk of floor(L/N) + 1",
     "        *shard_numel = (pos + N - 1) / N;",
     "        *shard_numel = pos / N + 1;"),
    ("PER_PARAM chunk of floor(d0/N) + 1 rows",
     "            int64_t rows = (dim0[i] + N - 1) / N;",
     "            int64_t rows = dim0[i] / N + 1;"),
    # pack / unpack
    ("PER_PARAM pack writes a rank's chunk column-major",
     "                        int64_t dst = (int64_t)r * c + off[i] + (row - lo) * in + col;",
     "                        int64_t dst = (int64_t)r * c + off[i] + col * rows[i] + (row - lo);"),
    ("PER_PARAM pack drops the final row of a short last chunk",
     "                if (hi > dim0[i]) hi = dim0[i];",
     "                if (hi > dim0[i]) hi = dim0[i] - 1;"),
    ("FLAT unpack reads rank-interleaved instead of rank-major",
     "                src_index = owner * c + local;",
     "                src_index = local * N + owner;"),
    ("PER_PARAM unpack reads a chunk column-major",
     "                src_index = owner * c + oi + local_row * in + col;",
     "                src_index = owner * c + oi + col * ci + local_row;"),
    # reduce-scatter
    ("reduce-scatter multiplies by 1/N instead of dividing by N",
     "            out[f] = acc / divisor;",
     "            out[f] = acc * (1.0f / divisor);"),
    ("reduce-scatter sums bf16 ranks in reverse order",
     "                acc = bf16_to_f32(((const uint16_t*)rank_bufs[0])[f]);\n"
     "                for (int r = 1; r < N; ++r) acc = acc + bf16_to_f32(((const uint16_t*)rank_bufs[r])[f]);",
     "                acc = bf16_to_f32(((const uint16_t*)rank_bufs[N - 1])[f]);\n"
     "                for (int r = N - 2; r >= 0; --r) acc = acc + bf16_to_f32(((const uint16_t*)rank_bufs[r])[f]);"),
    ("reduce-scatter sums fp32 ranks in reverse order",
     "                acc = ((const float*)rank_bufs[0])[f];\n"
     "                for (int r = 1; r < N; ++r) acc = acc + ((const float*)rank_bufs[r])[f];",
     "                acc = ((const float*)rank_bufs[N - 1])[f];\n"
     "                for (int r = N - 2; r >= 0; --r) acc = acc + ((const float*)rank_bufs[r])[f];"),
    # AdamW
    ("AdamW without the weight decay (plain Adam)",
     "        theta = theta - lr * weight_decay * theta;",
     "        theta = theta;"),
    ("Adam with L2 regularisation instead of decoupled decay",
     "        theta = theta - lr * weight_decay * theta;",
     "        g = g + weight_decay * theta;"),
    ("AdamW with beta1 and 1 - beta1 swapped",
     "        m = beta1 * m + (1.0 - beta1) * g;",
     "        m = (1.0 - beta1) * m + beta1 * g;"),
    ("AdamW second moment of |g| instead of g^2",
     "        v = beta2 * v + (1.0 - beta2) * g * g;",
     "        v = beta2 * v + (1.0 - beta2) * fabs(g);"),
    ("AdamW first-moment bias correction one step ahead",
     "    const double bc1 = 1.0 - pow(beta1, (double)step);",
     "    const double bc1 = 1.0 - pow(beta1, (double)(step + 1));"),
    ("AdamW without the first-moment bias correction",
     "        double mhat = m / bc1;",
     "        double mhat = m;"),
    ("AdamW without the second-moment bias correction",
     "        double vhat = v / bc2;",
     "        double vhat = v;"),
    ("AdamW with eps inside the square root",
     "        theta = theta - lr * mhat / (sqrt(vhat) + eps);",
     "        theta = theta - lr * mhat / sqrt(vhat + eps);"),
    # optimizer-state initialisation
    ("init: exp_avg left as it was, not zeroed",
     "        exp_avg[k] = 0.0f;",
     "        (void)exp_avg;"),
    ("init: exp_avg_sq left as it was, not zeroed",
     "        exp_avg_sq[k] = 0.0f;",
     "        (void)exp_avg_sq;"),
    ("init: master widened from the bf16's upper byte only",
     "        master[k] = elem_bytes == 2 ? bf16_to_f32(((const uint16_t*)param_shards)[k])",
     "        master[k] = elem_bytes == 2 ? bf16_to_f32(((const uint16_t*)param_shards)[k] & 0xFF00u)"),
    ("init: master as the integer value of the bf16 bits",
     "        master[k] = elem_bytes == 2 ? bf16_to_f32(((const uint16_t*)param_shards)[k])",
     "        master[k] = elem_bytes == 2 ? (float)((const uint16_t*)param_shards)[k]"),
    # accumulation
    ("accumulation returns the sum, not the mean, over micro-batches",
     "    for (int64_t f = 0; f < count; ++f) grad[f] = accum[f] / k;",
     "    for (int64_t f = 0; f < count; ++f) grad[f] = accum[f];"),
    # DDP
    ("DDP bucket closes only above the cap",
     "        if (fill >= cap_bytes) {",
     "        if (fill > cap_bytes) {"),
    ("DDP bucket count includes an empty trailing bucket",
     "    return fill > 0 ? bucket + 1 : bucket;",
     "    return bucket + 1;"),
    ("DDP buckets filled in registration order",
     "    for (int t = T - 1; t >= 0; --t) {",
     "    for (int t = 0; t < T; ++t) {"),
    ("DDP average sums ranks in reverse order",
     "            float acc = bf16_to_f32(grads[t][k]);\n"
     "            for (int r = 1; r < N; ++r) acc = acc + bf16_to_f32(grads[(size_t)r * (size_t)T + (size_t)t][k]);",
     "            float acc = bf16_to_f32(grads[(size_t)(N - 1) * (size_t)T + (size_t)t][k]);\n"
     "            for (int r = N - 2; r >= 0; --r) acc = acc + bf16_to_f32(grads[(size_t)r * (size_t)T + (size_t)t][k]);"),
    ("DDP average returns the sum over ranks",
     "            out[t][k] = f32_to_bf16_rne(acc / divisor);",
     "            out[t][k] = f32_to_bf16_rne(acc);"),
]


# The oracle's Python parts: (name, file under oracle/, exact text, replacement).
PY_MUTANTS = [
    ("ZeRO-1 resident bytes with one gradient copy fewer", "ledger.py",
     "        return 2 * P * b + P * bopt / N",
     "        return P * b + P * bopt / N"),
    ("ZeRO-2 resident bytes without the sharded gradient", "ledger.py",
     "        return P * b + P * (b + bopt) / N",
     "        return P * b + P * bopt / N"),
    ("ZeRO-3 resident bytes without the sharded gradient", "ledger.py",
     "        return P * (2 * b + bopt) / N",
     "        return P * (b + bopt) / N"),
    ("worst peak without the gathered parameter copy", "ledger.py",
     "        return resident + P * b",
     "        return resident"),
    ("FULL_SHARD traffic without the (N-1)/N factor", "ledger.py",
     "        return 3 * P * (N - 1) / N",
     "        return 3 * P"),
    ("SHARD_GRAD_OP / NO_SHARD traffic halved", "ledger.py",
     "        return 2 * P * (N - 1) / N",
     "        return P * (N - 1) / N"),
    ("LayerNorm backward without its second mean term", "dp_equivalence.py",
     "    do = rstd * (dxhat - dxhat.mean(axis=1, keepdims=True)\n"
     "                 - xhat * (dxhat * xhat).mean(axis=1, keepdims=True))",
     "    do = rstd * (dxhat - dxhat.mean(axis=1, keepdims=True))"),
    ("ReLU backward without the mask", "dp_equivalence.py",
     "    da = dh * (a > 0)",
     "    da = dh"),
    ("loss gradient of the sum, not the mean, over samples", "dp_equivalence.py",
     "    dy = diff / B",
     "    dy = diff"),
    ("unequal rank batches averaged without token weights", "dp_equivalence.py",
     "        w = (n_r / B) if token_weighted else (1.0 / N)",
     "        w = 1.0 / N"),
    ("micro-batch gradients summed, not averaged", "dp_equivalence.py",
     "            acc[k] += g[k] / micro_batches",
     "            acc[k] += g[k]"),
]

PY_CONTROL = ("control: Python oracle copied with nothing planted", "ledger.py",
              '"""Closed-form memory and communication ledgers of DP / ZeRO / FSDP.',
              '"""Closed-form memory and communication ledgers of DP / ZeRO / FSDP (control).')

# A "mutation" that changes nothing but a comment: built and run like the others.
CONTROL = ("control: no mistake planted",
           "/* Round a binary32 to the nearest bf16, ties to the even bf16.  Written from",
           "/* Round a binary32 to the nearest bf16, ties to the even bf16 (control).  Written from")


def _gcc_available():
    try:
        subprocess.run(["gcc", "--version"], check=True, capture_output=True)
        return True
    except Exception:
        return False


def _run_mutant(workdir, name, find, replace):
    """Build one mutant and run the pins against it: (pytest exit code, output)."""
    with open(SRC) as f:
        src = f.read()
    if src.count(find) != 1:
        return None, f"mutation target not unique or missing: {name}"
    os.makedirs(workdir, exist_ok=True)
    mutant_c = os.path.join(workdir, "ss_oracle_mutant.c")
    with open(mutant_c, "w") as f:
        f.write(src.replace(find, replace))
    lib = oracle.compile_library(mutant_c, os.path.join(workdir, "libssoracle_mutant.so"))
    env = dict(os.environ, **{oracle.ORACLE_LIB_ENV: lib, "OMP_NUM_THREADS": "2"})
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def _run_py_mutant(workdir, lib, name, relfile, find, replace):
    """Copy the oracle package, the workloads and the pin suite, plant one
    mistake in a Python file of the copied oracle, and run the pins there
    (against the unmodified C library): (pytest exit code, output)."""
    import shutil
    skip = shutil.ignore_patterns("__pycache__", "*.so", "*.pyc")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(workdir, "oracle"), ignore=skip)
    shutil.copytree(os.path.join(ROOT, "workloads"), os.path.join(workdir, "workloads"), ignore=skip)
    tdir = os.path.join(workdir, "tests")
    os.makedirs(tdir)
    for f in ("__init__.py", "conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(HERE, f), tdir)
    shutil.copytree(os.path.join(HERE, "golden"), os.path.join(tdir, "golden"))
    path = os.path.join(workdir, "oracle", relfile)
    with open(path) as f:
        src = f.read()
    if src.count(find) != 1:
        return None, f"mutation target not unique or missing: {name}"
    with open(path, "w") as f:
        f.write(src.replace(find, replace))
    env = dict(os.environ, **{oracle.ORACLE_LIB_ENV: lib, "OMP_NUM_THREADS": "2"})
    env.pop("PYTHONPATH", None)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(tdir, "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=workdir, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every mutant built and run against the pins, several at a time."""
    import concurrent.futures as cf
    base = tmp_path_factory.mktemp("mutants")
    workers = max(1, min(8, os.cpu_count() or 1))
    jobs = MUTANTS + [CONTROL]
    lib = oracle.build()
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = {m[0]: ex.submit(_run_mutant, str(base / f"m{i}"), *m) for i, m in enumerate(jobs)}
        for i, m in enumerate(PY_MUTANTS + [PY_CONTROL]):
            futs[m[0]] = ex.submit(_run_py_mutant, str(base / f"p{i}"), lib, *m)
        return {name: f.result() for name, f in futs.items()}


@pytest.mark.skipif(not _gcc_available(), reason="gcc is needed to build the mutants")
def test_unmutated_build_passes_the_pins(mutant_results):
    """The control: the same build and run with nothing planted passes, so a
    failing mutant run is the pins at work, not the harness."""
    code, out = mutant_results[CONTROL[0]]
    assert code == 0, out


@pytest.mark.skipif(not _gcc_available(), reason="gcc is needed to build the mutants")
def test_unmutated_python_copy_passes_the_pins(mutant_results):
    """The control for the Python mutants: the copied tree with nothing planted
    passes the pins, so a failing run is the pins at work, not the copy."""
    code, out = mutant_results[PY_CONTROL[0]]
    assert code == 0, out


@pytest.mark.skipif(not _gcc_available(), reason="gcc is needed to build the mutants")
@pytest.mark.parametrize("name", [m[0] for m in MUTANTS] + [m[0] for m in PY_MUTANTS])
def test_pins_catch_mutant(mutant_results, name):
    code, out = mutant_results[name]
    # exit code 1: the pins ran and at least one failed (a crash or a
    # collection error would give another code and would not show the pins
    # at work)
    assert code == 1, f"mutant survived the pins: {name}\n{out}"
