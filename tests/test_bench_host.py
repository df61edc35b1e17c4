"""Host-side pieces of bench.py that run without a GPU: the host description the CPU
baseline carries (Arm and x86 /proc/cpuinfo forms), and the reference arm (the oracle on the
host cores): its stepped timing and the JSON line it prints."""
import argparse
import builtins
import io
import json
import re

import bench

_ARM = ("processor\t: 0\nBogoMIPS\t: 2000.00\nFeatures\t: fp asimd\nCPU implementer\t: 0x41\n"
        "CPU architecture: 8\nCPU variant\t: 0x0\nCPU part\t: 0xd4f\nCPU revision\t: 0\n\n")
_X86 = "processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Some CPU @ 2.70GHz\nflags\t\t: fpu\n\n"


def _with_cpuinfo(monkeypatch, text):
    real_open = builtins.open

    def fake_open(path, *a, **k):
        if path == "/proc/cpuinfo":
            return io.StringIO(text)
        return real_open(path, *a, **k)

    monkeypatch.setattr(builtins, "open", fake_open)
    return bench._host_cpu()


def test_host_cpu_arm(monkeypatch):
    h = _with_cpuinfo(monkeypatch, _ARM)
    assert h["cpu"].startswith("Arm Neoverse V2") and h["nproc"] >= 1


def test_host_cpu_x86(monkeypatch):
    h = _with_cpuinfo(monkeypatch, _X86)
    assert h["cpu"].startswith("Some CPU @ 2.70GHz")


def test_host_cpu_unreadable(monkeypatch):
    def no_file(path, *a, **k):
        raise OSError("no cpuinfo")

    monkeypatch.setattr(builtins, "open", no_file)
    h = bench._host_cpu()
    assert isinstance(h["cpu"], str) and h["cpu"]


def test_reference_arm_times_exactly_k_steps_on_row_slices():
    """W untimed and exactly K timed steps; when K + W whole forwards do not fit the budget,
    each step runs the oracle on a slice of whole 64-row groups."""
    r = bench._oracle_spqr_steps(5, 3, budget_s=1e-6, N=1024, K=512)  # no host fits: one 64-row group
    m = re.match(r"5 timed steps after 3 warm-up, .* over (\d+) of the 1024x512 M=1 layer's rows", r["sample"])
    assert m, r["sample"]
    assert int(m.group(1)) == 64
    assert r["value"] > 0 and r["ms_per_step"] > 0 and r["kind"] == "oracle" and r["cores"] == 1
    r = bench._oracle_spqr_steps(2, 3, budget_s=1e6, N=1024, K=512)
    assert "over 1024 of the 1024x512" in r["sample"]  # the whole layer when it fits


def test_reference_arm_line(monkeypatch, capsys):
    calls = []
    fake = {"value": 0.04, "unit": "GB/s", "cores": 1, "kind": "oracle", "ms_per_step": 550.0, "sample": "s"}

    def fake_subprocess(extra=()):
        calls.append(list(extra))
        return fake

    monkeypatch.setattr(bench, "cpu_baseline_subprocess", fake_subprocess)
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(argparse.Namespace(steps=7, warmup=4))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert calls == [["--steps", "7", "--warmup", "4"]]
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["steps"] == 7 and line["warmup"] == 4 and line["ms_per_step"] == 550.0
    assert line["value"] == 0.04 and line["higher_is_better"] is True and line["n_gpus"] == 1
    assert line["cpu_baseline"] == fake
    assert line["e2e"] == {"value": 0.04, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"] == bench._config(1)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setattr(bench, "cpu_baseline_subprocess", lambda extra=(): (_ for _ in ()).throw(AssertionError))
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(argparse.Namespace(steps=7, warmup=4))
    assert capsys.readouterr().out == ""


def test_oracle_row_slice_equals_the_rows_of_the_whole_layer():
    """The reference arm's steps rest on this: the oracle's dequantization of a row slice of
    the canonical arrays is bit for bit the same rows of the whole layer's (rows with and
    without outliers, a slice starting and ending mid-layer)."""
    import numpy as np

    import qlin_synth as synth
    from oracle import spqr

    N, K = 256, 1024
    W, _ = synth.spqr_layer(N, K, 1, seed=5)
    p = spqr.pack(W, 0.02)
    full = spqr.dequantize_canonical(N, K, p["codes"], p["qs_bits"], p["qz_bits"], p["stats"], p["rowptr"], p["col"],
                                     p["val"])
    rp = np.asarray(p["rowptr"])
    for r0, r1 in [(0, 64), (64, 192), (192, 256), (17, 18)]:
        a, b = int(rp[r0]), int(rp[r1])
        part = spqr.dequantize_canonical(r1 - r0, K, p["codes"][r0:r1], p["qs_bits"][r0:r1], p["qz_bits"][r0:r1],
                                         p["stats"][r0:r1], rp[r0:r1 + 1] - a, p["col"][a:b], p["val"][a:b])
        assert np.array_equal(part.view(np.uint32), full[r0:r1].view(np.uint32)), (r0, r1)
    assert int(rp[-1]) > 0
