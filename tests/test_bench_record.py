"""The benchmark's DRAM-traffic record (profiles/tc_splitk_traffic.txt): the
hash of the kernel's code that keys it, and when bench.py reports it as
roofline.traffic (no GPU needed)."""
import hashlib
import os

import bench


def test_code_of_drops_comments_and_blank_lines_only():
    src = 'int a = 1; // one\n\n/* two\n lines */ int b = 2;\nconst char *s = "// kept /* too */";\n'
    assert bench.code_of(src) == 'int a = 1;\n int b = 2;\nconst char *s = "// kept /* too */";'


def _record(tmp_path, sources, ops, cut="", constants_only=""):
    h = hashlib.sha256()
    for name in sources:
        text = bench.code_of((tmp_path / name).read_text())
        if cut and cut in text:
            text = text[:text.index(cut)]
        if name in constants_only.split():
            text = "\n".join(line for line in text.splitlines() if line.startswith("constexpr"))
        h.update(text.encode())
    (tmp_path / "profiles").mkdir(exist_ok=True)
    lines = ["# a test record", f"sources = {' '.join(sources)}", f"code_sha256 = {h.hexdigest()}",
             f"ops_per_launch = {ops}", "dram_bytes_per_launch = 4096"]
    if cut:
        lines.append(f"device_code_ends_at = {cut}")
    if constants_only:
        lines.append(f"constants_only = {constants_only}")
    (tmp_path / "profiles" / "tc_splitk_traffic.txt").write_text("\n".join(lines) + "\n")


def test_traffic_record_keys(tmp_path, monkeypatch):
    """Reported while the device code and the header's constants hash to the
    record and a launch computes as many operations; comment edits and host
    code after the marker do not matter; a device-code or constant change, or
    another number of operations per launch, drops it."""
    (tmp_path / "k.cu").write_text("__global__ void k() { int x = 1; }\n__global__ void end_mark() {}\nint host() { return 1; }\n")
    (tmp_path / "h.h").write_text("constexpr int kA = 4;\nint host_decl();\n")
    _record(tmp_path, ["k.cu", "h.h"], 8, cut="__global__ void end_mark", constants_only="h.h")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic(8) == 4096
    assert bench.kernel_traffic(1) is None
    # comments, host code after the marker and the header's other lines may change
    (tmp_path / "k.cu").write_text("// note\n__global__ void k() { int x = 1; }\n__global__ void end_mark() {}\n"
                                   "int host() { return 2; }\n")
    (tmp_path / "h.h").write_text("constexpr int kA = 4;\nint host_decl(int);\n")
    assert bench.kernel_traffic(8) == 4096
    # the device code or a constant may not
    (tmp_path / "h.h").write_text("constexpr int kA = 5;\nint host_decl(int);\n")
    assert bench.kernel_traffic(8) is None
    (tmp_path / "h.h").write_text("constexpr int kA = 4;\n")
    (tmp_path / "k.cu").write_text("__global__ void k() { int x = 2; }\n__global__ void end_mark() {}\n")
    assert bench.kernel_traffic(8) is None


def test_committed_record_is_well_formed():
    """The committed record names existing sources and carries the keys the
    bench reads."""
    path = os.path.join(bench.ROOT, "profiles", "tc_splitk_traffic.txt")
    rec = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
    for key in ("sources", "code_sha256", "ops_per_launch", "dram_bytes_per_launch"):
        assert key in rec, key
    for src in rec["sources"].split():
        assert os.path.exists(os.path.join(bench.ROOT, src)), src
    assert int(rec["dram_bytes_per_launch"]) > 0 and int(rec["ops_per_launch"]) >= 1
