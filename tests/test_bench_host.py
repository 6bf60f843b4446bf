"""Host-side logic of bench.py that needs no GPU: the algorithmic byte count behind
the roofline, the lookup of recorded DRAM traffic (valid only while the kernel's
source is unchanged), the clock and throttle-reason summary of nvidia-smi samples,
and the number of input copies that keeps timed inputs out of L2."""
import hashlib
import os

import bench


def test_step_bytes_counts_every_operand_once():
    # INT4 codes K*N/2, one bf16 scale per 128 weights along K, bf16 A [M, K] and Y [M, N]
    K, N = 4096, 14336
    for M, want in ((1, 30_314_496), (4, 30_425_088), (16, 30_867_456)):
        codes = (K // 8) * N * 4                 # int32 [K/8, N]
        scales = (K // 128) * N * 2              # bf16 [K/128, N]
        assert bench.step_bytes(M) == codes + scales + M * K * 2 + M * N * 2 == want


def _fake_tree(tmp_path, source: bytes, recorded_hash: str):
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "bit_quantized_linear_quantizers_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "kern.cu").write_bytes(source)
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel workload bytes file hash\n"
        f"my_kernel   wl_a   1234567   kern.cu   {recorded_hash}\n"
        f"my_kernel   wl_b   7654321   kern.cu   {recorded_hash}   # trailing comment\n",
        encoding="utf-8")
    return csrc / "kern.cu"


def test_kernel_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = b"__global__ void my_kernel() {}\n"
    h = hashlib.sha256(src).hexdigest()[:16]
    path = _fake_tree(tmp_path, src, h)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("my_kernel", "wl_a") == 1234567.0
    assert bench.kernel_traffic("my_kernel", "wl_b") == 7654321.0
    assert bench.kernel_traffic("my_kernel", "wl_c") is None
    assert bench.kernel_traffic("other_kernel", "wl_a") is None
    path.write_bytes(src + b"// changed\n")       # counters taken on an older source: no figure
    assert bench.kernel_traffic("my_kernel", "wl_a") is None
    path.unlink()
    assert bench.kernel_traffic("my_kernel", "wl_a") is None


def test_kernel_traffic_without_a_record(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("my_kernel", "wl_a") is None


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    s.out = "\n".join(lines)
    return s


def test_clock_summary_median_max_and_reasons():
    idle = "Not Active"
    lines = [
        f"0, 2070, 2070, 900.1, 0x0, {idle}, {idle}, {idle}, {idle}",
        f"0, 1980, 2070, 1390.0, 0x4, {idle}, {idle}, {idle}, Active",
        f"0, 2070, 2070, 1200.0, 0x0, {idle}, {idle}, {idle}, {idle}",
        "garbage line",
        f"0, [N/A], 2070, 1.0, 0x0, {idle}, {idle}, {idle}, {idle}",
    ]
    got = _sampler_with(lines).summary()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_each_slowdown_kind():
    a, n = "Active", "Not Active"
    lines = [f"0, 1500, 2070, 1000, 0x8, {a}, {n}, {n}, {n}",
             f"0, 1400, 2070, 1000, 0x8, {n}, {a}, {n}, {n}",
             f"0, 1300, 2070, 1000, 0x8, {n}, {n}, {a}, {n}"]
    got = _sampler_with(lines).summary()
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert got["sm_mhz"] == 1400.0 and got["samples"] == 3


def test_clock_summary_without_samples():
    assert _sampler_with([]).summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}


def test_copies_exceed_twice_l2():
    l2 = 126 << 20
    for nbytes in (1, 4 << 20, 30_314_496, l2, 3 * l2):
        c = bench.copies_for(nbytes, l2)
        assert c >= 2
        assert c * nbytes >= 2 * l2 or c == 2
        assert c == 2 or (c - 1) * nbytes < 2 * l2        # no more copies than needed


def test_host_cpu_model(tmp_path):
    x86 = tmp_path / "x86"
    x86.write_text("processor\t: 0\nvendor_id\t: GenuineIntel\nmodel\t\t: 167\n"
                   "model name\t: Example CPU @ 2.70GHz\n\nprocessor\t: 1\nmodel name\t: other\n")
    got = bench.host_cpu(str(x86))
    assert got["cpu"] == "Example CPU @ 2.70GHz" and got["nproc"] >= 1
    arm = tmp_path / "arm"
    arm.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\n"
                   "CPU variant\t: 0x0\nCPU part\t: 0xd4f\nCPU revision\t: 0\n")
    assert bench.host_cpu(str(arm))["cpu"] == "implementer 0x41 part 0xd4f"
    assert bench.host_cpu(str(tmp_path / "missing"))["cpu"]          # falls back to the platform


def test_oracle_timing_pins_one_core_and_restores():
    before = os.sched_getaffinity(0)
    with bench._one_core() as core:
        assert core in before and os.sched_getaffinity(0) == {core}
    assert os.sched_getaffinity(0) == before


def _recorded_commands():
    """(file, ncu command, bench arguments) for every command recorded under profiles/."""
    import glob
    import re
    import shlex
    out = []
    for path in sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*"))):
        text = open(path, encoding="utf-8").read()
        text = re.sub(r"\\\n\s*(#\s*)?", " ", text)                  # join continued lines
        for line in text.splitlines():
            line = line.lstrip("# ").strip()
            if line.startswith("ncu ") and "python bench.py" in line:
                argv = shlex.split(line.split("python bench.py", 1)[1])
                out.append((os.path.basename(path), line, argv))
    return out


def test_recorded_profile_commands_run_committed_files():
    """Every ncu command recorded under profiles/ keeps the clocks unlocked and runs
    bench.py with arguments its parser still accepts."""
    cmds = _recorded_commands()
    assert len({f for f, _, _ in cmds}) >= 3, "fewer recorded profiling commands than expected"
    for fname, line, argv in cmds:
        assert "--clock-control none" in line, fname
        args = bench.build_parser().parse_args(argv)
        assert args.warmup >= 3, fname
        assert set(args.rows.split(",")) <= set(bench.ROW_NAMES), fname
