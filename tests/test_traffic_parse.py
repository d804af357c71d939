"""CPU check of the DRAM-traffic accounting of a profiled step (host logic only):
a synthetic ncu launch list in the CSV format ncu writes, parsed into the fused
and unfused steps' bytes with each step's write-back pass."""
from gemm_epilogue_transformer_tmem_gb300 import traffic

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
          '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')


def _rows(i, name, read, write, us, ru="Mbyte", wu="Mbyte"):
    base = f'"{i}","1","python","h","{name}","1","7","(256, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics"'
    return [f'{base},"dram__bytes_read.sum","{ru}","{read}"', f'{base},"dram__bytes_write.sum","{wu}","{write}"',
            f'{base},"gpu__time_duration.sum","usecond","{us}"']


def _csv(seq):
    lines = ["==PROF== Connected to process 1", HEADER]
    for i, (name, r, w, us) in enumerate(seq):
        lines += _rows(i, name, r, w, us)
    return "\n".join(lines) + "\n"


FILL = "void at::native::vectorized_elementwise_kernel<4, at::native::FillFunctor<float>>(int, T2, T3)"
RED = "void at::native::reduce_kernel<512, 1, at::native::ReduceOp<float>>(T3)"


def test_steps_and_write_back():
    g = "void coda::coda_gemm_epilogue_kernel<false, true, false, true, coda::EpiFixed<4>, false, false>(CUtensorMap)"
    seq = [(FILL, 0, 268, 30), (RED, 268, 100, 40),          # warm-up flush
           (g, 50, 10, 80),                                   # warm-up step
           (FILL, 0, 268, 30), (RED, 268, 120, 40),
           (g, 51, 11, 81), ("void coda::finalize_rows_kernel(float)", 1, 0.5, 2),   # fused step
           (RED, 268, 60, 40),                                # its write-back: 60 MB
           (FILL, 0, 268, 30), (RED, 268, 100, 40),
           ("void coda::rmsnorm_kernel(int)", 17, 16, 9), ("void coda::coda_gemm_epilogue_kernel<x>(CUtensorMap)", 60, 20, 90),
           (RED, 268, 50, 40)]                                # unfused write-back: 50 MB
    launches = traffic.read_launches(_csv(seq))
    assert len(launches) == len(seq)
    entry, md = traffic.summarize("rmsproj", launches, "ncu ...")
    assert entry["fused_step_read"] == 52_000_000
    assert entry["fused_step_write"] == 71_500_000          # 11 + 0.5 + 60 MB
    assert entry["fused_writeback"] == 60_000_000
    assert entry["unfused_step_bytes"] == (17 + 60 + 16 + 20 + 50) * 1_000_000
    assert entry["dominant_kernel_bytes"] == 62_000_000
    assert entry["dominant_kernel"].startswith("void coda::coda_gemm_epilogue_kernel")
    assert "write-back" in md and "ncu ..." in md


def test_units_and_dominant_call_of_a_chain():
    g = "coda::coda_gemm_epilogue_kernel"
    seq = [(FILL, 0, 1, 1), (RED, 1, 0, 1)]
    seq += [(f"{g}<{k}>(CUtensorMap)", 10 * (k + 1), 1, 1) for k in range(4)]
    seq += [(RED, 1, 5, 1), (FILL, 0, 1, 1), (RED, 1, 0, 1), ("coda::rmsnorm_kernel", 2, 2, 1), (RED, 1, 7, 1)]
    text = _csv(seq).replace('"Mbyte","40"', '"Gbyte","0.04"')   # the same value in another unit
    launches = traffic.read_launches(text)
    entry, _ = traffic.summarize("llama", launches)
    # llama's dominant call is the third GEMM of the step (the up-projection)
    assert entry["dominant_kernel_bytes"] == 31_000_000
    assert entry["fused_step_read"] == 100_000_000
    assert entry["fused_step_write"] == 9_000_000
    assert entry["unfused_step_bytes"] == 11_000_000


def test_kernel_hash_is_stable():
    assert traffic.kernel_hash() == traffic.kernel_hash()
    assert len(traffic.kernel_hash()) == 16


def test_launch_shares():
    seq = [("coda::a_kernel(int)", 0, 0, 30.0), ("coda::b_kernel(int)", 0, 0, 10.0), ("coda::a_kernel(int)", 0, 0, 60.0)]
    md = traffic.launch_shares(traffic.read_launches(_csv(seq)), "ncu ...")
    assert "| `coda::a_kernel` | 2 | 90.0 | 90.0% |" in md
    assert "| `coda::b_kernel` | 1 | 10.0 | 10.0% |" in md
