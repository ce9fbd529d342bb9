"""HostPipeline's argument checks run before any device memory is touched (no GPU needed)."""
import pytest

from linear_attention_05_gb300.pipeline import HostPipeline


@pytest.mark.parametrize("n_seq,seq_len,groups,parts", [
    (4, 4096, 3, 1),    # groups must divide the sequences
    (4, 4096, 2, 2),    # time slices need one sequence per group
    (4, 4096, 4, 3),    # slices must divide the sequence
    (4, 4000, 4, 2),    # ... into multiples of 64 tokens
])
def test_rejects_bad_grouping(n_seq, seq_len, groups, parts):
    with pytest.raises(ValueError):
        HostPipeline(n_seq, seq_len, 2, 128, 128, device="cpu", groups=groups, parts=parts)
