"""Host logic of the bench's launch units: which calls of a step run as one program launch (no GPU)."""
import os

import bench
import workloads as wl


def _names(calls, units):
    return [calls[u].name if isinstance(u, int) else (u[0], [calls[i].name for i in u[1]]) for u in units]


def test_default_step_groups_the_small_calls_into_one_launch():
    w = bench.workloads_by_key()[bench.DEFAULT_WORKLOAD]
    calls = list(w.calls)
    units = bench.launch_groups(calls, w.layers, 152)
    # the largest call keeps its own launch, first; then one batch of the other calls of at least one row per SM;
    # then one program launch of the small calls (84 rows: one wave of the mixed variant)
    assert units[0] == 1 and calls[1].name == "swiglu_q8_dynamic_T2048_I53248"
    assert [u[0] for u in units[1:]] == ["batch", "bf16+fp8"]
    assert units[1][1] == [0] + [i for i, c in enumerate(calls) if c.T == 1000]
    small = [i for i, c in enumerate(calls) if c.T < 152]
    assert units[2][1] == small                                       # every small call once, in list order
    assert {(calls[i].kind, calls[i].mode) for i in small} == {
        ("add_rmsnorm", None), ("swiglu", None), ("add_rmsnorm_q8", "static"), ("swiglu_q8", "dynamic")}
    # without batches, every unit sits where its first call stood
    units = bench.launch_groups(calls, w.layers, 152, batches=False)
    flat = [u if isinstance(u, int) else u[1][0] for u in units]
    assert flat == sorted(flat) and [u[0] for u in units if not isinstance(u, int)] == ["bf16+fp8"]


def test_classes_split_when_their_rows_exceed_one_per_sm():
    d = wl.N01
    calls = [wl.Call("add_rmsnorm", 100, 1024, d), wl.Call("swiglu_q8", 60, 1024, d, mode="dynamic"),
             wl.Call("swiglu", 10, 1024, d)]
    assert bench.launch_groups(calls, 1, 152) == [("bf16", [0, 2]), ("fp8", [1])]
    assert bench.launch_groups(calls, 1, 200) == [("bf16+fp8", [0, 1, 2])]


def test_programs_take_no_dynamic_norm():
    d = wl.N01
    calls = [wl.Call("add_rmsnorm_q8", 4, 1024, d, mode="static"), wl.Call("add_rmsnorm_q8", 4, 1024, d, mode="dynamic"),
             wl.Call("swiglu_q8", 4, 1024, d, mode="dynamic"), wl.Call("swiglu_q8", 4, 1024, d, mode="static"),
             wl.Call("swiglu_nvfp4", 4, 1024, d), wl.Call("add_rmsnorm", 4, 1024, d)]
    units = bench.launch_groups(calls, 1, 152)
    assert units == [("bf16+fp8", [0, 2, 3, 5]), 1, ("nvfp4", [4])]


def test_no_grouping_across_layers_wide_norms_or_allreduce():
    d = wl.N01
    calls = [wl.Call("add_rmsnorm", 1, 1536, d), wl.Call("swiglu", 1, 8960, d)]
    assert bench.launch_groups(calls, 28, 152) == [0, 1]              # layers share a residual: keep the sequence
    wide = [wl.Call("add_rmsnorm", 1, 16384, d), wl.Call("swiglu", 1, 53248, d)]
    assert bench.launch_groups(wide, 1, 152) == [0, ("bf16", [1])]    # the program holds norms up to 8192 wide
    ar = [wl.Call("allreduce_rmsnorm", 2, 4096, d, partials=2), wl.Call("add_rmsnorm", 2, 4096, d)]
    assert bench.launch_groups(ar, 1, 152) == [0, ("bf16", [1])]
    assert bench.launch_groups(calls, 1, 1, batches=False) == [0, 1]  # nothing below one row per SM


def test_batches_take_every_call_of_one_row_per_sm_but_the_largest():
    d = wl.N01
    calls = [wl.Call("add_rmsnorm", 152, 1024, d), wl.Call("swiglu", 1215, 1024, d), wl.Call("swiglu", 4000, 1024, d),
             wl.Call("swiglu_q8", 500, 1024, d, mode="dynamic"), wl.Call("add_rmsnorm_nvfp4", 300, 1024, d),
             wl.Call("swiglu", 5, 1024, d)]
    assert bench.launch_groups(calls, 1, 152) == [2, ("batch", [0, 1, 3, 4]), ("bf16", [5])]
    assert bench.launch_groups(calls, 1, 152, max_batch=3) == [2, ("batch", [0, 1, 3]), ("batch", [4]), ("bf16", [5])]
    assert bench.launch_groups(calls[:3], 1, 152) == [2, ("batch", [0, 1])]
    assert bench.launch_groups(calls[1:3], 1, 152) == [0, 1]           # one call besides the largest: no batch
    assert bench.launch_groups(calls[:5], 28, 152) == [0, 1, 2, 3, 4]  # layers share buffers: no batch
    assert bench.launch_groups(calls, 1, 152, batches=False) == [0, 1, 2, 3, 4, ("bf16", [5])]
    ar = [wl.Call("add_rmsnorm", 2000, 4096, d), wl.Call("allreduce_rmsnorm", 400, 4096, d, partials=2),
          wl.Call("add_rmsnorm", 300, 4096, d)]
    assert bench.launch_groups(ar, 1, 152) == [0, 1, 2]               # the all-reduce norm is no batch op


def test_groups_split_at_the_op_limit():
    d = wl.N01
    calls = [wl.Call("swiglu", 1 + i, 256, d) for i in range(10)]
    units = bench.launch_groups(calls, 1, 152, max_ops=4)
    assert units == [("bf16", [0, 1, 2, 3]), ("bf16", [4, 5, 6, 7]), ("bf16", [8, 9])]


def test_traffic_hash_ignores_comments_and_layout_but_not_code(tmp_path, monkeypatch):
    """A recorded DRAM traffic figure stays valid while the kernel's sources change only in comments or layout,
    and is dropped (hash mismatch) when code changes."""
    import shutil
    root = tmp_path / "repo"
    for sub in ("include", "memory_bound_decoder_gb300/csrc", "memory_bound_decoder_gb300/tuning"):
        shutil.copytree(os.path.join(bench.ROOT, sub), root / sub)
    monkeypatch.setattr(bench, "ROOT", str(root))
    call = next(c for w in bench.workloads_by_key().values() for c in w.calls if c.kind == "swiglu_q8")
    base = bench.kernel_src_hash(call)
    src = root / "memory_bound_decoder_gb300/csrc/swiglu.cu"
    text = src.read_text()
    src.write_text(text.replace("namespace mbd {", "// a new comment\n/* and a block\n   comment */\n\n  namespace mbd {", 1))
    assert bench.kernel_src_hash(call) == base
    src.write_text(text.replace("namespace mbd {", "namespace mbd { constexpr int kUnused = 1;", 1))
    assert bench.kernel_src_hash(call) != base
    src.write_text(text)
    norm = root / "memory_bound_decoder_gb300/csrc/norm.cu"   # another kernel's source: no effect
    norm.write_text(norm.read_text() + "\nstatic int unused_norm_symbol;\n")
    assert bench.kernel_src_hash(call) == base
