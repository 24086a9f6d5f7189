"""The adaptive switch of the rollout loop ("SAM投机推理：长序列强化学习训练加速利器"
§3.1.1): drafting only while at most `threshold` requests are active."""
from sam_drafting_verification_gb300.rollout import speculation_k


def test_speculation_only_at_or_below_the_threshold():
    assert speculation_k(8, 8, 3) == 3
    assert speculation_k(9, 8, 3) == 0
    assert speculation_k(1, 8, 3) == 3
    assert speculation_k(500, None, 3) == 3  # no threshold: always
    assert speculation_k(4, 8, 0) == 0       # K = 0: plain decoding
