"""Host-side logic of bench.py that decides what a run reports (CPU only): the
clock summary that accepts or rejects a run, the kernel fingerprint that ties a
profiled DRAM traffic figure to the code it was measured on, and the lookup of
that figure."""
import os

import bench

BUS = "00000009:01:00.0"


def _sample(bus, sm, reasons=("Not Active",) * 4):
    return ", ".join(["2026/12/02 10:00:00.000", bus, str(sm), "2070", "900.0", *reasons]) + "\n"


def test_clock_summary_filters_the_gpu_and_collects_reasons():
    lines = [_sample(BUS, 2070), _sample(BUS, 2055),
             _sample(BUS, 1980, ("Not Active", "Not Active", "Not Active", "Active")),
             _sample("00000019:01:00.0", 900, ("Active",) * 4),     # another GPU
             "garbage line\n", _sample(BUS, "[N/A]")]
    c = bench.summarise_clocks(lines, BUS.lower())
    assert c["samples"] == 3 and c["sm_mhz"] == 2055 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    hot = bench.summarise_clocks([_sample(BUS, 1500, ("Active", "Not Active", "Active", "Not Active"))], BUS)
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.summarise_clocks([], BUS)["samples"] == 0


def _tree(tmp_path, code):
    for f in bench.KERNEL_SOURCES:
        p = tmp_path / f
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text(code.get(f, "int x;\n"))
    return tmp_path


def test_fingerprint_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    f0 = bench.KERNEL_SOURCES[0]
    monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path, {f0: "int a = 1; // one\n/* x */ int b;\n"})))
    base = bench.kernel_fingerprint()
    (tmp_path / f0).write_text("int a = 1;   // another comment\n\n/* a\\nlonger one */ int b;\n")
    assert bench.kernel_fingerprint() == base
    (tmp_path / f0).write_text("int a = 2; // one\n/* x */ int b;\n")
    assert bench.kernel_fingerprint() != base


def test_profiled_traffic_needs_a_matching_fingerprint(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path, {})))
    (tmp_path / "profiles").mkdir()
    fp = bench.kernel_fingerprint()
    prof = tmp_path / "profiles" / "qnorm_rope_kv_insert_stress.md"
    prof.write_text(f"Kernel sources fingerprint: `{fp}`\n\ntraffic_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("stress") == 1234
    prof.write_text("Kernel sources fingerprint: `0000000000000000`\n\ntraffic_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("stress") is None
    assert bench.profiled_traffic("decode") is None   # no summary at all


def test_committed_summaries_name_their_commands():
    """Every ncu summary gives the command that made it, and that command runs only
    committed files (bench.py with flags)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name in os.listdir(os.path.join(root, "profiles")):
        text = open(os.path.join(root, "profiles", name)).read()
        assert "ncu " in text and "--clock-control none" in text, name
        assert "python bench.py" in text, name
        assert "_work" not in text, name


def test_self_check_flags_rates_above_the_copy_ceiling():
    assert bench.self_check(6500.0, 6510.0, 6630.0, 6400.0) == {"ok": True, "over_copy_ceiling": 0.9819}
    bad = bench.self_check(7200.0, 7300.0, 6630.0, 6400.0)
    assert not bad["ok"] and bad["over_copy_ceiling"] > 1.05


def test_cpu_model_is_a_nonempty_name():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_cpulist_round_trip():
    assert bench._cpulist("0-3,8,10-11\n") == [0, 1, 2, 3, 8, 10, 11]
    assert bench._ranges([11, 0, 1, 2, 3, 8, 10]) == "0-3,8,10-11"
    assert bench._cpulist("") == [] and bench._ranges([]) == ""


def test_pages_by_node_finds_the_mapping_of_an_address(tmp_path, monkeypatch):
    maps = ("00400000 default file=/bin/x mapped=3 N0=3\n"
            "7f0000000000 default anon=10 dirty=10 N0=4 N1=6 kernelpagesize_kB=64\n"
            "7f0000100000 default anon=2 N1=2\n")
    real_open = open

    def fake_open(path, *a, **kw):
        if path == "/proc/self/numa_maps":
            p = tmp_path / "numa_maps"
            p.write_text(maps)
            return real_open(p, *a, **kw)
        return real_open(path, *a, **kw)

    monkeypatch.setattr("builtins.open", fake_open)
    assert bench.pages_by_node(0x7f0000000040) == {0: 4, 1: 6}
    assert bench.pages_by_node(0x7f0000100000) == {1: 2}
    assert bench.pages_by_node(0x100) == {}


def test_counter_captures_run_small_cases():
    """A committed ncu command that collects more than the launch times (sections, sets
    or other metrics) must run a case that holds at most a few GB on the device: for
    the fused step, at most 3 GB of q (stress and bf16_store only with --tokens)."""
    import re
    import shlex
    from synth import configs
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name in os.listdir(os.path.join(root, "profiles")):
        text = open(os.path.join(root, "profiles", name)).read().replace("\\\n", " ")
        for line in text.splitlines():
            if "ncu " not in line or "python bench.py" not in line:
                continue
            ncu_part, bench_part = line.split("python bench.py", 1)
            metrics = re.findall(r"--metrics\s+(\S+)", ncu_part)
            times_only = (not re.search(r"--set|--section", ncu_part)
                          and all(m == "gpu__time_duration.sum" for m in metrics))
            if times_only:
                continue
            args = shlex.split(bench_part)
            get = lambda flag, default: args[args.index(flag) + 1] if flag in args else default
            op, wl = get("--op", "fused"), configs.WORKLOADS[get("--workload", "stress")]
            tokens = int(get("--tokens", wl.T))
            if op in ("fused", "prenorm"):
                assert tokens * wl.H * 1024 <= 3e9, (name, line.strip())
