"""CPU oracle (test infrastructure only): see oracle/joint_attn.py."""
