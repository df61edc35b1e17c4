"""Host-side pieces of bench.py that run without a GPU: the host description the CPU
baseline carries (Arm and x86 /proc/cpuinfo forms)."""
import builtins
import io

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
