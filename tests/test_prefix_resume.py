"""Resume arithmetic for cached prefixes (host only) and host-side checks of the
checkpointed prefill entry point."""
import ctypes

import pytest

import linear_attention_serving_chunkwise_gb300 as kda
from linear_attention_serving_chunkwise_gb300.build import build
from linear_attention_serving_chunkwise_gb300.prefix_resume import plan_resume


def test_resume_on_hash_and_checkpoint_boundaries():
    # 512-token hash blocks, snapshots every 512 tokens: boundaries are multiples of 512
    assert plan_resume(5000, 6000) == (4608, 8, 6000 - 4608)
    assert plan_resume(511, 6000) == (0, -1, 6000)
    assert plan_resume(512, 6000) == (512, 0, 5488)
    # a fully matched prompt still recomputes its last block's tokens
    assert plan_resume(4096, 4096).boundary == 3584
    # snapshots every 1024 tokens: only every second hash boundary is reusable
    assert plan_resume(5000, 6000, checkpoint_interval=1024) == (4096, 3, 1904)
    # snapshots every 192 tokens (lcm with 512 is 1536)
    assert plan_resume(5000, 6000, checkpoint_interval=192).boundary == 4608
    # limited slots
    assert plan_resume(5000, 6000, checkpoint_slots=4) == (2048, 3, 3952)
    # a 6144-token physical block does not move the KDA boundary
    assert plan_resume(6143, 12288).boundary == 5632


def test_resume_rejects_bad_arguments():
    with pytest.raises(ValueError):
        plan_resume(10, 5)
    with pytest.raises(ValueError):
        plan_resume(10, 20, checkpoint_interval=100)


def test_checkpointed_entry_validates_on_host():
    build()
    lib = kda.load()
    d = kda.make_desc(1, 256, 2, 64, 64, kda.KDA_F32)
    f = lambda a: ctypes.c_void_p(a)
    args = lambda interval, slots, ck: (ctypes.byref(d), f(0x10000), f(0x20000), f(0x30000), f(0x40000),
                                        f(0x50000), None, None, f(0x60000), None, interval, slots, ck, None, 0, None)
    assert lib.kda_prefill_checkpointed(*args(100, 2, f(0x900000))) == kda.KDA_ERR_INVALID_ARG   # not x64
    assert lib.kda_prefill_checkpointed(*args(128, 0, f(0x900000))) == kda.KDA_ERR_INVALID_ARG   # no slots
    assert lib.kda_prefill_checkpointed(*args(128, 2, None)) == kda.KDA_ERR_INVALID_ARG          # no buffer
    assert lib.kda_prefill_checkpointed(*args(128, 2, f(0x60000))) == kda.KDA_ERR_INVALID_ARG    # overlaps out
