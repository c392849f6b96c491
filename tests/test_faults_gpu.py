"""Bounded waits: a test makes every in-kernel wait run out (the producers withhold their
loads, a flag nothing else sets) and checks that the call reports PA_ERR_DEVICE_TIMEOUT,
that no GPU fault happens, and that the next call on the same context is correct.  The
cases reach the decode kernel, the prefill kernel, the head-dim-512 decode kernel, the
head-dim-256 prefill kernel and the persistent (work-list) decode mode."""
import pytest

from paged_kv_varlen_flashattention_gb300 import binding, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def _layout(name):
    if name == "prefill_d256":  # the head-dim-256 tensor-core prefill kernel
        return workloads.make_layout("faults_pf256", "bf16", [200, 90], [200, 300], num_heads=8, num_heads_k=2,
                                     head_dim=256, page_block_size=64, seed=21, spare=0.1)
    if name == "work_list":  # 20 sequences, one split: the persistent decode mode
        sk = [300 + 17 * b for b in range(20)]
        sk[7] = 20000
        return workloads.make_layout("faults_worklist", "bf16", [1] * 20, sk, num_heads=8, num_heads_k=2,
                                     head_dim=128, page_block_size=32, seed=22, spare=0.1)
    return workloads.small(name)


@pytest.mark.parametrize("name", ["decode", "prefill", "d512", "prefill_d256", "work_list"])
def test_wait_runs_out_and_context_survives(name):
    lay = _layout(name)
    inp = workloads.materialize(lay, device="cuda")
    binding.set_wait_limit_ns(20_000_000)  # 20 ms
    binding.set_withhold_loads(True)
    try:
        _gpu_call(inp)
        st = binding.device_status()
    finally:
        binding.set_withhold_loads(False)
        binding.set_wait_limit_ns(0)
    assert binding.STATUS[st] == "PA_ERR_DEVICE_TIMEOUT", binding.last_error()
    assert binding.device_status() == 0
    ref_o, ref_l = _gpu.oracle_for(inp.to("cpu"))
    out, lse = _gpu.run_cuda(inp)
    _gpu.compare(lay, out, lse, ref_o, ref_l)


def _gpu_call(inp):
    lay = inp.layout
    binding.varlen_fwd(inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.block_table,
                       max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k,
                       softmax_scale=lay.softmax_scale, window_left=lay.window_left,
                       window_right=lay.window_right)
