"""CPU oracle (test infrastructure only): see oracle.py and nvfp4_oracle.c."""
