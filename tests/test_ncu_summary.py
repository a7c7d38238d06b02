"""The ncu summariser reads both CSV forms ncu prints: the launch list
(details page, one row per launch and metric) and the raw page of a capture
(a header, a units row, one row per launch), with ncu's unit prefixes."""
import json

from paged_kv_cache_314_gb300 import ncu_summary as ns

DETAILS = "\n".join([
    "==PROF== Connected to process 1",
    '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
    '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
    '"Metric Value"',
    '"0","1","python3.12","h","void at::vectorized_elementwise_kernel<4, at::FillFunctor<int>, '
    'std::array<char *, 1>>(int, T2, T3)","1","7","(128, 1, 1)","(1, 1, 1)","0","10.3",'
    '"Command line profiler metrics","gpu__time_duration.sum","ns","2000"',
    '"1","1","python3.12","h","pa::<unnamed>::kv_write_kernel(pa::<unnamed>::KvWriteParams)",'
    '"1","7","(256, 1, 1)","(256, 1, 1)","0","10.3","Command line profiler metrics",'
    '"gpu__time_duration.sum","us","3.5"',
    '"2","1","python3.12","h","void pa::decode_persistent_kernel<__half, 128, 1, 0, __half>'
    '(pa::DecodeParams)","1","7","(160, 1, 1)","(760, 1, 1)","0","10.3",'
    '"Command line profiler metrics","gpu__time_duration.sum","us","196.5"',
    '"3","1","python3.12","h","void pa::decode_persistent_kernel<__half, 128, 1, 0, __half>'
    '(pa::DecodeParams)","1","7","(160, 1, 1)","(760, 1, 1)","0","10.3",'
    '"Command line profiler metrics","gpu__time_duration.sum","msecond","0.1985"',
    "==PROF== Disconnected from process 1",
])

RAW = "\n".join([
    '"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum",'
    '"lts__t_sector_hit_rate.pct","gpu__time_duration.sum","launch__registers_per_thread"',
    '"","","Gbyte","Mbyte","%","us",""',
    '"0","void decode_persistent_kernel<__half, 128, 1, 0, __half>(DecodeParams)","1.347173",'
    '"6.350848","0.228809","198.144000","72"',
    '"1","void decode_merge_rows_kernel<__half, 128>(DecodeParams)","5.943","0","24.99",'
    '"7.104","62"',
])


def test_launch_list_per_kernel():
    s = ns.summarise_launches(DETAILS, "cmd")
    k = s["kernels"]
    assert list(k) == ["decode_persistent_kernel", "kv_write_kernel",
                       "vectorized_elementwise_kernel"]
    assert k["decode_persistent_kernel"]["launches"] == 2
    assert abs(k["decode_persistent_kernel"]["total_s"] - 395.0e-6) < 1e-12
    assert abs(k["kv_write_kernel"]["total_s"] - 3.5e-6) < 1e-15
    assert abs(sum(v["share"] for v in k.values()) - 1.0) < 1e-12


def test_raw_page_counters_and_traffic(tmp_path):
    s = ns.summarise_kernel(RAW, "decode_persistent", "llama7b", "cmd", "simt")
    (launch,) = s["launches"]
    assert launch["dram_bytes_read"] == 1.347173e9
    assert launch["dram_bytes_write"] == 6.350848e6
    assert s["traffic_bytes_per_launch"] == 1347173000 + 6350848
    assert abs(launch["duration_s"] - 198.144e-6) < 1e-12
    assert s["l2_hit_rate_pct"] == 0.228809
    assert s["kernel"] == "decode_persistent_kernel"
    assert s["kernel_sources"] == list(ns.KERNEL_SOURCES["simt"])
    assert s["kernel_source_sha256_16"] == ns.kernel_source_hash(ns.KERNEL_SOURCES["simt"])
    out = tmp_path / "x.json"
    csv_path = tmp_path / "raw.csv"
    csv_path.write_text(RAW)
    ns.main(["kernel", "--csv", str(csv_path), "--kernel", "merge_rows", "--family", "simt",
             "--out", str(out)])
    assert json.loads(out.read_text())["traffic_bytes_per_launch"] == 5943000000  # Gbyte column


def test_short_names():
    assert ns._short("void pa::decode_persistent_kernel<__half, 128, 1, 0, __half>"
                     "(pa::DecodeParams)") == "decode_persistent_kernel"
    assert ns._short("pa::<unnamed>::kv_write_kernel(pa::<unnamed>::KvWriteParams)") == \
        "kv_write_kernel"
    assert ns._short("void pa::(anonymous namespace)::prefix_widen_kernel<__nv_bfloat16>"
                     "(pa::DecodeParams, __nv_bfloat16 *, __nv_bfloat16 *, int *)") == \
        "prefix_widen_kernel"
    assert ns._short("void unnamed>::prefix_widen_kernel<__nv_bfloat16>(DecodeParams, T1 *, T1 *, "
                     "int *)") == "prefix_widen_kernel"
